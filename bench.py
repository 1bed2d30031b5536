#!/usr/bin/env python3
"""Benchmark of the tree-verify hot path on one GB300 per rank.

One step = ancestors (a1) + tree attention (a2) + greedy verify (a3) + KV
commit (a4) for the whole batch of one layer, back to back on one stream
(plus the best-first tree build a5 for the budgeted-tree workloads).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload 70b]
  python bench.py --impl reference ...   # the CPU oracle arm

Prints ONE JSON line (rank 0).  Inputs are synthetic (seeded, the shapes of
the named workload) and resident in HBM before timing; L2 is flushed between
timed steps (a 256 MiB write, then a 256 MiB read of another buffer, so the
step starts cold with no dirty lines to write back), outside the timed
events.  Under
torchrun every rank runs its own replica (sequences are independent units;
no data-path collective): value = all ranks' steps / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import gen  # noqa: E402

METRIC = "tree-verify steps/s (attn+accept+commit) and achieved HBM GB/s vs GB300 peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
FLUSH_BYTES = 256 << 20
DESCRIPTIONS = {
    "tiny": "tiny verify layer: B=1, Hq=Hkv=4, D=64, prefix 128, 15-node random tree, V=1000",
    "8b": "Llama-3-8B-shaped verify layer: B=1, Hq=32, Hkv=8, D=128, prefix 4096, 63-node static "
          "tree (depth 6), V=128256",
    "ragged": "batched ragged verify layer: B=16, Hq=32, Hkv=8, D=128, prefix U[512,8192], "
              "31-node random trees (depth<=5), V=32000",
    "70b": "long-context 70B-shaped verify layer: B=4, Hq=64, Hkv=8, D=128, prefix 32768, "
           "127-node random trees (depth<=8), V=128256, paged cache with shuffled 16-token blocks",
}


def workload_inputs(name, batch=None):
    """Host arrays for a workload (numpy), and a description.  batch: keep the
    first `batch` sequences only (the same shapes at a smaller size, for
    profiling)."""
    if name.startswith("bastion"):
        N = int(name[len("bastion"):])
        q, root = gen.bastion_marginals()
        return ("bastion", N, q, root), ("BASTION-style budgeted tree: B=8, K=16, V=32000 "
                                         "marginals, best-first budget N=%d, verify on Hq=32, "
                                         "Hkv=8, D=128, prefix 2048" % N)
    if name == "dynamic":
        c = gen.DYNAMIC
        return ("dynamic", c), ("EAGLE-2-style dynamic draft tree: B=%d, V=%d, top-%d expansion "
                                "over %d levels (drafter rows resident), rerank to N=%d, verify "
                                "on Hq=32, Hkv=8, D=128, prefix 2048"
                                % (c["B"], c["V"], c["k"], c["levels"], c["N"]))
    inp = gen.verify_workload(name)
    if batch is not None and batch < inp.B:
        return (gen.first_sequences(inp, batch),
                DESCRIPTIONS[name] + " (first %d of %d sequences)" % (batch, inp.B))
    return inp, DESCRIPTIONS[name]


def algorithmic_bytes(inp, moved_total):
    """Per-kernel algorithmic bytes of one step (what each kernel must move at
    least once)."""
    B, N, Hq, Hkv, D, V, Dm = inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, inp.V, inp.D_max
    W = (N + 31) // 32
    slots = int((inp.prefix_len.astype(np.int64) + inp.n_nodes).sum())
    a1 = 4 * (B * N + B + B * (N + 1) * (Dm + 1) + B * N + B * N * W + B)
    a2 = 4 * Hkv * D * slots + 4 * B * N * Hq * D + 4 * B * N * Hq
    a3 = 4 * B * N * V
    a4 = 8 * Hkv * D * int(moved_total)
    return {"tree_build_ancestors": a1, "tree_attn_fwd": a2, "tree_verify_greedy": a3,
            "kv_commit_path": a4}


def tree_depths(parent_row, n):
    """Depth of every node of one parent array (root depth 0)."""
    d = np.zeros(n, dtype=np.int64)
    for i in range(n):
        j, k = i, 0
        while parent_row[j] >= 0:
            j = int(parent_row[j])
            k += 1
        d[i] = k
    return d


def attention_flops(inp):
    """Algorithmic FLOPs of one tree_attn_fwd launch: each (node, q head) row
    takes a D-long dot product and a D-long weighted sum (2 FLOPs per
    multiply-add each) over the keys it sees, its prefix plus its ancestor
    path (itself included)."""
    keys = 0
    for b in range(inp.B):
        nb = int(inp.n_nodes[b])
        keys += int(inp.prefix_len[b]) * nb + int((tree_depths(inp.parent[b], nb) + 1).sum())
    return 4.0 * inp.D * inp.Hq * keys


def load_tensor_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s bf16 burst, one earlier GB300 measurement)"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)", pk
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)", {}


def _code_only(text):
    """C/C++/CUDA source with comments removed and every run of whitespace
    collapsed to one space; string and character literals are kept as they
    are (inline PTX lives in them)."""
    out, i, n = [], 0, len(text)
    while i < n:
        ch = text[i]
        if ch in "\"'":
            j = i + 1
            while j < n and text[j] != ch:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(ch)
            i += 1
    return " ".join("".join(out).split())


# The sources each profiled kernel is built from (its translation unit and the
# headers that unit includes); a kernel's profile figures are tied to these.
KERNEL_SOURCES = {
    "tree_attn_fwd": ["attention.cu", "sm100_ptx.cuh", "tsd_common.cuh"],
    "tree_verify_greedy": ["verify.cu", "commit_core.cuh", "sm100_ptx.cuh", "tsd_common.cuh"],
    "best_first_tree_build": ["best_first.cu", "sm100_ptx.cuh", "tsd_common.cuh"],
}


def kernel_sources_digest(kernel_key=None):
    """Digest of the CUDA sources' code (comments and layout ignored), so
    profile figures stay attached to the kernels they were taken on: of the
    sources of one profiled kernel (KERNEL_SOURCES), or of every source."""
    csrc = os.path.join(ROOT, "tree_speculative_decoding_virtual_gb300", "csrc")
    names = sorted(KERNEL_SOURCES[kernel_key] if kernel_key else os.listdir(csrc))
    h = hashlib.sha256()
    for f in names:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_key, workload):
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken on
    the kernel's current sources."""
    path = os.path.join(ROOT, "profiles", "traffic_%s_%s.md" % (kernel_key, workload))
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    d = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not d or d.group(1) != kernel_sources_digest(kernel_key):
        return None
    return float(m.group(1))


class ClockSampler:
    def __init__(self, index):
        self.proc = None
        fd, self.path = tempfile.mkstemp(prefix="tsd_clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index),
                 "--query-gpu=timestamp,clocks.sm,clocks.max.sm,power.draw,"
                 "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
                 "clocks_event_reasons.hw_thermal_slowdown,"
                 "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        self.marks = []

    def mark(self):
        self.marks.append(time.time())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        try:
            os.unlink(self.path)
        except OSError:
            pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v == "Active"})
        loaded = [r[0] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and reference arm)
# ---------------------------------------------------------------------------

ORACLE_CHILD = r"""
import json, os, sys, time
sys.path.insert(0, %(root)r)
import numpy as np
import gen, oracle
name, steps, frac = %(name)r, %(steps)d, %(frac)f
inp = gen.verify_workload(name)
rng = np.random.default_rng(0)
rows = [(b, i, h) for b in range(inp.B) for i in range(int(inp.n_nodes[b])) for h in range(inp.Hq)]
pick = rng.choice(len(rows), size=max(1, int(round(frac * len(rows)))), replace=False)
sample = [rows[j] for j in sorted(pick)]
c = inp.cache
t_attn = t_rest = 0.0
for s in range(steps):
    t0 = time.perf_counter()
    anc, depth, mask, err = oracle.build_ancestors(inp.parent, inp.n_nodes, inp.D_max)
    t1 = time.perf_counter()
    out, lse = oracle.tree_attention(inp.q, c.k, c.v, c.block_table, inp.prefix_len, inp.n_nodes,
                                     inp.parent, err, inp.scale, sample=sample)
    t2 = time.perf_counter()
    am, A, leaf, path, bonus = oracle.verify_greedy(inp.logits, inp.tokens, inp.parent,
                                                    inp.n_nodes, err, inp.D_max)
    k1, v1, nl, mv = oracle.commit_path(c.k, c.v, c.block_table, inp.prefix_len, A, path, err)
    t3 = time.perf_counter()
    t_attn += t2 - t1
    t_rest += (t1 - t0) + (t3 - t2)
per_step_full = (t_rest + t_attn / (len(sample) / len(rows))) / steps
print(json.dumps({"sec_per_full_step": per_step_full, "steps": steps, "sample_rows": len(sample),
                  "total_rows": len(rows), "wall": t_attn + t_rest}))
"""


def run_oracle_child(name, steps, frac, threads):
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(threads)
    code = ORACLE_CHILD % {"root": ROOT, "name": name, "steps": steps, "frac": frac}
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                       timeout=1800)
    if r.returncode != 0:
        raise RuntimeError("oracle child failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


def oracle_sample_fraction(name):
    # attention rows evaluated per oracle step (the rest of the step runs in full)
    return {"tiny": 1.0, "8b": 0.125, "ragged": 0.05, "70b": 0.004}.get(name, 0.05)


def cpu_baseline(name, budget_steps=3, single_thread=True):
    threads = os.cpu_count() or 1
    frac = oracle_sample_fraction(name)
    res = run_oracle_child(name, budget_steps, frac, threads)
    value = 1.0 / res["sec_per_full_step"]
    one = None
    if single_thread:
        r1 = run_oracle_child(name, 1, frac, 1)
        one = {"value": 1.0 / r1["sec_per_full_step"], "unit": "steps/s", "cores": 1}
    return {"value": value, "unit": "steps/s", "cores": threads, "kind": "oracle",
            "single_thread": one,
            "sample": "%d oracle steps of the %s workload; each runs ancestors, verify and commit "
                      "in full and attention on %d of %d (seq, node, q-head) rows, scaled to the "
                      "full row count" % (res["steps"], name, res["sample_rows"],
                                           res["total_rows"])}


# ---------------------------------------------------------------------------
# multi-rank aggregation (replicas: every rank runs the whole workload)
# ---------------------------------------------------------------------------

def max_over_ranks(value: float, world: int, device="cpu") -> float:
    """The slowest rank's time: every rank contributes its own, rank 0 reports
    the max (the job is done when the last replica is)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(ms_per_step_max: float, world: int) -> float:
    """Steps per second of the whole job: all ranks' steps over the max time."""
    return world * 1000.0 / ms_per_step_max


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

# the configurations measured beside the headline workload in one run
CONFIG_SET = ["tiny", "8b", "ragged", "70b", "bastion16", "bastion32", "bastion64", "bastion128",
              "bastion256"]


def _graph_capture(torch, fn):
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    with torch.cuda.graph(g):
        fn()
    return g


def measure_workload(name, args, rank, world, dev, flush_l2, full, verify="greedy"):
    """Set up one workload on the device and time it.  One step = the hot
    path over the whole batch, captured as one CUDA graph.  Returns the
    result dict (rank 0) or None."""
    import torch
    import torch.distributed as dist

    import tree_speculative_decoding_virtual_gb300 as tsd

    stream = torch.cuda.current_stream()
    steps, warmup = args.steps, args.warmup
    w, desc = workload_inputs(name, getattr(args, "batch", None))
    bastion = isinstance(w, tuple) and w[0] == "bastion"
    dynamic = isinstance(w, tuple) and w[0] == "dynamic"

    def T(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if dtype is not None:
            t = t.view(dtype)
        return t.to(dev)

    if bastion:
        _, N_b, q_marg, root = w
        qd, rootd = T(q_marg), T(root)
        bf_ws = torch.empty(tsd.best_first_workspace_bytes(*q_marg.shape, N_b), dtype=torch.uint8,
                            device=dev)
        bf_out = [torch.empty((q_marg.shape[0], N_b), dtype=torch.int32, device=dev) for _ in range(3)]
        rho = torch.empty((q_marg.shape[0], N_b), dtype=torch.float32, device=dev)
        ahat = torch.empty((q_marg.shape[0],), dtype=torch.float64, device=dev)
        tsd.best_first_tree_build(qd, rootd, N_b, *bf_out, rho, ahat, workspace=bf_ws)
        torch.cuda.synchronize()
        par_h, tok_h, dep_h = [x.cpu().numpy() for x in bf_out]
        top1 = np.argmax(q_marg, axis=-1)  # input synthesis only: plants target choices
        inp = gen.bastion_verify_inputs(par_h, tok_h, dep_h, top1)
    elif dynamic:
        # The drafter's rows for every level's frontier are generated once on
        # the host (seeded per node) and kept in HBM; the timed step runs the
        # level-by-level expansion on them, the rerank, and a1-a4 on the tree.
        dc = w[1]
        dB, dV, dk, dL, dN = dc["B"], dc["V"], dc["k"], dc["levels"], dc["N"]
        dM = tsd.dynamic_tree_pool_size(dL, dk)
        d_pool = tsd.dynamic_tree_new_pool(dB, dM, dev)
        d_root = T(np.random.default_rng(dc["seed"]).integers(0, dV, size=dB).astype(np.int32))
        d_fr = [None] + [torch.empty((dB, dk), dtype=torch.int32, device=dev) for _ in range(dL)]
        d_ws = torch.empty(tsd.dynamic_tree_workspace_bytes(dB, dk, dk), dtype=torch.uint8,
                           device=dev)
        d_rows = []
        fr_h = np.zeros((dB, 1), dtype=np.int32)
        for level in range(1, dL + 1):
            rows = np.stack([gen.dynamic_draft_rows(dc["seed"], b, fr_h[b], dV, dc["temp"])
                             for b in range(dB)])
            d_rows.append(T(rows))
            tsd.dynamic_tree_expand(d_rows[-1], dk, level, d_pool, root_token=d_root,
                                    frontier=d_fr[level - 1], next_frontier=d_fr[level],
                                    workspace=d_ws)
            fr_h = d_fr[level].cpu().numpy()
        d_tree = [torch.empty((dB, dN), dtype=torch.int32, device=dev) for _ in range(3)]
        d_score = torch.empty((dB, dN), dtype=torch.float32, device=dev)
        tsd.dynamic_tree_rerank(d_pool, dM, dN, *d_tree, d_score)
        torch.cuda.synchronize()
        par_h, tok_h, dep_h = [x.cpu().numpy() for x in d_tree]
        inp = gen.dynamic_verify_inputs(par_h, tok_h, dep_h)
    else:
        inp = w

    B, N, Hq, Hkv, D, V, Dm = inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, inp.V, inp.D_max
    c = inp.cache
    stochastic = verify == "stochastic"
    if stochastic:
        q_draft_h, tok_h, ua_h, ud_h = gen.stochastic_for(inp)
        inp.tokens = tok_h
        q_draft, u_acc, u_drw = T(q_draft_h), T(ua_h), T(ud_h)
        del q_draft_h
    parent, n_nodes, prefix = T(inp.parent), T(inp.n_nodes), T(inp.prefix_len)
    tokens, logits, q = T(inp.tokens), T(inp.logits), T(inp.q, torch.bfloat16)
    if dynamic:  # a1-a4 read the tree the rerank writes every step
        parent, tokens = d_tree[0], d_tree[1]
    table = T(c.block_table)
    kc, vc = T(c.k, torch.bfloat16), T(c.v, torch.bfloat16)
    max_slots = int((inp.prefix_len + inp.n_nodes).max())
    W = (N + 31) // 32
    i32 = dict(dtype=torch.int32, device=dev)
    anc = torch.empty((B, N + 1, Dm + 1), **i32)
    depth = torch.empty((B, N), **i32)
    mask = torch.empty((B, N, W), **i32)
    err = torch.empty((B,), **i32)
    out = torch.empty((B, N, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, N, Hq), dtype=torch.float32, device=dev)
    attn_need = tsd.tree_attn_workspace_bytes(B, N, Hq, Hkv, D, max_slots)
    attn_ws = (torch.empty((attn_need,), dtype=torch.uint8, device=dev) if attn_need > 0 else None)
    ver_ws = torch.zeros((tsd.tree_verify_workspace_bytes(B, N, V),), dtype=torch.uint8, device=dev)
    st_ws = (torch.zeros((tsd.tree_verify_stochastic_workspace_bytes(B, N, V),), dtype=torch.uint8,
                         device=dev) if stochastic else None)
    am = torch.empty((B, N), **i32)
    drw = torch.empty((B, N), **i32)
    A = torch.empty((B,), **i32)
    leaf = torch.empty((B,), **i32)
    path = torch.empty((B, Dm + 1), **i32)
    bonus = torch.empty((B,), **i32)
    new_len = torch.empty((B,), **i32)
    moved = torch.empty((B,), **i32)
    status = torch.zeros((1,), **i32)

    verify_name = "tree_verify_stochastic" if stochastic else "tree_verify_greedy"
    fused_name = "tree_verify_greedy_commit"
    head = ((["best_first_tree_build"] if bastion else [])
            + (["dynamic_tree_expand", "dynamic_tree_rerank"] if dynamic else [])
            + ["tree_build_ancestors", "tree_attn_fwd"])
    # every entry point is timed on its own; the greedy step runs verification
    # and commit as the one fused launch
    names = head + [verify_name, "kv_commit_path"] + ([] if stochastic else [fused_name])
    step_names = head + ([verify_name, "kv_commit_path"] if stochastic else [fused_name])
    attn_launches = tsd.tree_attn_launches(B, N, Hq, Hkv, D, max_slots)
    launches_per_step = ((2 if bastion else 0) + (2 * dL + 1 if dynamic else 0) + 1
                         + attn_launches + (2 if stochastic or B == 1 else 1))

    calls = {}
    if bastion:
        calls["best_first_tree_build"] = lambda: tsd.best_first_tree_build(
            qd, rootd, N_b, *bf_out, rho, ahat, workspace=bf_ws)
    if dynamic:
        def expand_all():
            for level in range(1, dL + 1):
                tsd.dynamic_tree_expand(d_rows[level - 1], dk, level, d_pool, root_token=d_root,
                                        frontier=d_fr[level - 1], next_frontier=d_fr[level],
                                        workspace=d_ws)
        calls["dynamic_tree_expand"] = expand_all
        calls["dynamic_tree_rerank"] = lambda: tsd.dynamic_tree_rerank(
            d_pool, dM, dN, *d_tree, d_score)
    calls["tree_build_ancestors"] = lambda: tsd.tree_build_ancestors(
        parent, n_nodes, Dm, anc, depth, mask, err)
    calls["tree_attn_fwd"] = lambda: tsd.tree_attn_fwd(
        q, kc, vc, table, prefix, n_nodes, mask, err, max_slots, out=out, lse=lse,
        workspace=attn_ws, status=status)
    calls["tree_verify_greedy"] = lambda: tsd.tree_verify_greedy(
        logits, tokens, parent, anc, depth, mask, n_nodes, err, Dm, am, A, leaf, path, bonus,
        workspace=ver_ws)
    if stochastic:
        calls["tree_verify_stochastic"] = lambda: tsd.tree_verify_stochastic(
            logits, q_draft, tokens, parent, n_nodes, err, u_acc, u_drw, Dm, am, drw, A, leaf,
            path, bonus, workspace=st_ws)
    calls["kv_commit_path"] = lambda: tsd.kv_commit_path(
        kc, vc, table, prefix, n_nodes, A, path, err, N, Dm, new_len=new_len, moved=moved,
        status=status)
    calls[fused_name] = lambda: tsd.tree_verify_greedy_commit(
        logits, tokens, parent, anc, depth, mask, n_nodes, err, Dm, kc, vc, table, prefix,
        argmax=am, accept_len=A, leaf=leaf, path=path, bonus=bonus, new_len=new_len, moved=moved,
        status=status, workspace=ver_ws)

    def step():
        for n in step_names:
            calls[n]()

    for _ in range(warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    moved_total = int(moved.sum().item())
    assert int(status.item()) == 0, "device status %d" % int(status.item())
    rejected_rows = internal_rows = leaf_draws = 0
    if stochastic:
        # rows the method must read: the target row of every internal node
        # (its children are decided on it), the draft row of each node that
        # saw a rejection, and the target row of the walk's last node when it
        # is a leaf (the bonus is drawn there); other leaves need nothing
        nx = am.cpu().numpy()
        leaf_h = leaf.cpu().numpy()
        for b in range(B):
            nb = int(inp.n_nodes[b])
            for i in range(nb):
                kids = [j for j in range(1, nb) if int(inp.parent[b, j]) == i
                        and 0 <= int(inp.tokens[b, j]) < V]
                if kids:
                    internal_rows += 1
                    if nx[b, i] != kids[0]:
                        rejected_rows += 1
                elif i == int(leaf_h[b]):
                    leaf_draws += 1

    # CUDA graphs: the whole step; each entry point alone; each entry point
    # behind the L2 flush inside the graph, and the flush alone (their
    # difference is the entry point's device time from the end of the flush,
    # without the gap between the start event and a graph's first kernel)
    capture = lambda fn: _graph_capture(torch, fn)
    g_step = capture(step)
    g_one = {n: capture(calls[n]) for n in names}
    g_flush = capture(flush_l2)

    def flushed(fn):
        def run():
            flush_l2()
            fn()
        return run
    g_fk = {n: capture(flushed(calls[n])) for n in names}
    g_fstep = capture(flushed(step))
    torch.cuda.synchronize()

    sampler = ClockSampler(int(dev.index or 0)) if (rank == 0 and full) else None
    # ---- timed region 1: whole steps (the headline value) ----
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for s_ in range(steps):
        flush_l2()
        ev[s_][0].record(stream)
        g_step.replay()
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    ms_per_step = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / steps, world, dev)
    clocks = sampler.stop() if sampler else None

    # ---- timed region 2: per entry point ----
    reps = max(3, min(steps, 400))
    nev = len(names) + 1
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(reps)]
    torch.cuda.synchronize()
    for s_ in range(reps):
        flush_l2()
        kev[s_][0].record(stream)
        for j, n in enumerate(names):
            g_one[n].replay()
            kev[s_][j + 1].record(stream)
    torch.cuda.synchronize()
    per_entry = {n: 0.0 for n in names}
    for e in kev:
        for j, n in enumerate(names):
            per_entry[n] += e[j].elapsed_time(e[j + 1])
    entry_us = {n: 1000.0 * v / reps for n, v in per_entry.items()}

    # ---- timed region 3: kernel-only device time (graph deltas) ----
    order = ["flush"] + names + ["step"]
    graphs = dict(g_fk, flush=g_flush, step=g_fstep)
    acc = {n: 0.0 for n in order}
    for _ in range(reps):
        for n in order:
            a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a_.record(stream)
            graphs[n].replay()
            b_.record(stream)
            b_.synchronize()
            acc[n] += a_.elapsed_time(b_)
    flush_us = 1000.0 * acc["flush"] / reps
    kernel_us = {n: max(0.0, 1000.0 * acc[n] / reps - flush_us) for n in names}
    step_kernel_us = max(0.0, 1000.0 * acc["step"] / reps - flush_us)

    stacked_us = n_layers = None
    if full:
        # ---- a4 layer-stacked: the step's accepted paths committed into L
        # layers' caches in one launch (bandwidth is only meaningful this way;
        # per layer the commit moves a few KB).  L = 80, or fewer when 80
        # layers of this cache would take more than 4 GB.
        layer_bytes = 2 * kc.numel() * kc.element_size()
        n_layers = int(max(1, min(80, (4 << 30) // max(layer_bytes, 1))))
        kL = kc.unsqueeze(0).repeat(n_layers, 1, 1, 1, 1)
        vL = vc.unsqueeze(0).repeat(n_layers, 1, 1, 1, 1)
        stacked = lambda: tsd.kv_commit_path(kL, vL, table, prefix, n_nodes, A, path, err, N, Dm,
                                             new_len=new_len, moved=moved, status=status)
        stacked()
        g_stacked = capture(stacked)
        torch.cuda.synchronize()
        sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(max(3, min(steps, 200)))]
        for a_, b_ in sev:
            flush_l2()
            a_.record(stream)
            g_stacked.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        stacked_us = 1000.0 * sum(a_.elapsed_time(b_) for a_, b_ in sev) / len(sev)
        del kL, vL, g_stacked

    e2e = None
    if full:
        # ---- e2e: host buffers through the public API, copies inside the timing ----
        h_in = {"q": q, "logits": logits, "parent": parent, "tokens": tokens, "n_nodes": n_nodes,
                "prefix_len": prefix}
        if stochastic:
            h_in.update({"q_draft": q_draft, "u_accept": u_acc, "u_draw": u_drw})
        if dynamic:  # the drafter's rows are the inputs; the tree is built on the device
            del h_in["parent"], h_in["tokens"]
            h_in.update({"draft_rows_%d" % (i + 1): r for i, r in enumerate(d_rows)})
        pinned = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in h_in.items()}
        for k, v in h_in.items():
            pinned[k].copy_(v.cpu())
        h_out_src = {"out": out, "argmax": am, "accept_len": A, "leaf": leaf, "path": path,
                     "bonus": bonus, "new_len": new_len}
        if stochastic:
            h_out_src["draw"] = drw
        h_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                 for k, v in h_out_src.items()}
        h2d = sum(v.numel() * v.element_size() for v in pinned.values())
        d2h = sum(v.numel() * v.element_size() for v in h_out.values())
        e2e_steps = max(3, min(steps, 200))
        e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                  for _ in range(e2e_steps)]
        # The logits (and the stochastic verifier's draft rows and uniforms)
        # are read only by the verify call, so they are copied on a second
        # stream while the tree and attention kernels run, as a serving loop
        # would overlap them; that stream starts after the start event and
        # after the previous step's last reads, and verify waits for it.
        late = [k for k in h_in if k in ("logits", "q_draft", "u_accept", "u_draw")]
        copy_stream = torch.cuda.Stream()
        # When a step's inputs are more than twice L2 they sweep it on their
        # own, so steps run back to back with no flush, as a serving loop runs
        # them: a step's late inputs are copied as soon as the previous step's
        # verify has read the buffers, under the previous step's commit and
        # result copies and this step's tree and attention kernels, and the
        # whole run is timed.  Smaller inputs keep the flush between steps and
        # a timed region per step.
        pipelined = h2d > FLUSH_BYTES  # the flush buffer is about twice L2
        # Greedy tree workloads also keep two sets of input buffers, used by
        # alternate steps, so that the next step's copies need not wait for
        # this step's verify.
        double = pipelined and not (bastion or dynamic or stochastic)
        bufs = [h_in, {k: torch.empty_like(v) for k, v in h_in.items()}] if double else [h_in]
        read_ev = [None, None]  # per buffer set: its last step's verify has read it
        run_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        for s_ in range(e2e_steps + 3):
            bi = s_ % len(bufs)
            if double:  # the API calls read these names
                h_in = bufs[bi]
                q, logits, parent = h_in["q"], h_in["logits"], h_in["parent"]
                tokens, n_nodes, prefix = h_in["tokens"], h_in["n_nodes"], h_in["prefix_len"]
            if not pipelined:
                flush_l2()
            if s_ >= 3:
                if pipelined:
                    if s_ == 3:
                        run_ev[0].record(stream)
                else:
                    e2e_ev[s_ - 3][0].record(stream)
            if pipelined and read_ev[bi] is not None:
                copy_stream.wait_event(read_ev[bi])
            else:
                copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                if pipelined:
                    # the small inputs first, on the same stream, so that they
                    # do not queue behind the logits for the host link
                    for k, v in h_in.items():
                        if k not in late:
                            v.copy_(pinned[k], non_blocking=True)
                    small_ev = torch.cuda.Event()
                    small_ev.record(copy_stream)
                for k in late:
                    h_in[k].copy_(pinned[k], non_blocking=True)
            if pipelined:
                stream.wait_event(small_ev)
            else:
                for k, v in h_in.items():
                    if k not in late:
                        v.copy_(pinned[k], non_blocking=True)
            for n in step_names:  # the public API calls, launched from Python
                if n in (verify_name, fused_name):
                    stream.wait_stream(copy_stream)
                calls[n]()
                if n in (verify_name, fused_name):  # the last call that reads the inputs
                    read_ev[bi] = torch.cuda.Event()
                    read_ev[bi].record(stream)
            for k, v in h_out_src.items():
                h_out[k].copy_(v, non_blocking=True)
            if s_ >= 3 and not pipelined:
                e2e_ev[s_ - 3][1].record(stream)
        if pipelined:
            run_ev[1].record(stream)
        torch.cuda.synchronize()
        if pipelined:
            e2e_ms = max_over_ranks(run_ev[0].elapsed_time(run_ev[1]) / e2e_steps, world, dev)
        else:
            e2e_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in e2e_ev) / e2e_steps, world,
                                    dev)
        # the box's pinned host-to-device copy rate, for reading the e2e figure
        big = max(v.numel() * v.element_size() for v in pinned.values())
        src = max(pinned.values(), key=lambda v: v.numel() * v.element_size())
        dst = torch.empty_like(src, device=dev)
        hev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(20)]
        for a_, b_ in hev:
            a_.record(stream)
            dst.copy_(src, non_blocking=True)
            b_.record(stream)
        torch.cuda.synchronize()
        h2d_gbs = big / (min(a_.elapsed_time(b_) for a_, b_ in hev) * 1e-3) / 1e9
        e2e = {"value": round(whole_job_rate(e2e_ms, world), 2), "unit": "steps/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(e2e_ms, 4),
               "overlap": ("every input copied on a second stream (the small ones first, then %s) "
                           "into one of two buffer sets used by alternate steps, once the step "
                           "before the previous one has read that set, so copies run back to "
                           "back under the kernels; steps back to back (inputs > 2x L2), the run "
                           "timed whole"
                           if double else
                           "every input copied on a second stream once the previous step's "
                           "verify has read the inputs (the small ones first, then %s), under "
                           "its commit and result copies and this step's tree and attention "
                           "kernels; steps back to back (inputs > 2x L2), the run timed whole"
                           if pipelined else
                           "%s copied on a second stream under the kernels before verify; "
                           "L2 flushed between steps, each step timed") % "+".join(late),
               "pinned_h2d_gbs": round(h2d_gbs, 1),
               "pinned_h2d_probe": "one %d-byte pinned host-to-device copy, best of 20" % big}

    if rank != 0:
        return None
    peak, peak_src, _ = load_peaks()
    abytes = algorithmic_bytes(inp, moved_total)
    if stochastic:
        # every valid node's target row, the draft rows of nodes that saw a
        # rejection, and the per-node uniforms, tokens and parents
        abytes["tree_verify_stochastic"] = (4 * V * (internal_rows + rejected_rows + leaf_draws)
                                            + 4 * 4 * B * N)
        del abytes["tree_verify_greedy"]
    if dynamic:
        # each level reads its frontier's draft rows once
        abytes["dynamic_tree_expand"] = sum(4 * r.numel() for r in d_rows)
    if not stochastic:
        abytes[fused_name] = abytes["tree_verify_greedy"] + abytes["kv_commit_path"]
    step_bytes = sum(abytes.values())
    dom = max(["tree_attn_fwd", verify_name], key=lambda n: kernel_us[n])
    attn_flops = attention_flops(inp)
    tc_peak, tc_src = load_tensor_peak()
    # the attention's binding roof: HBM when its bytes take longer at peak
    # bandwidth than its FLOPs at peak tensor throughput, else the tensor pipe
    attn_tensor = attn_flops / (tc_peak * 1e12) > abytes["tree_attn_fwd"] / (peak * 1e9)
    tensor_bound = dom == "tree_attn_fwd" and attn_tensor
    t_dom = kernel_us[dom] * 1e-6
    achieved = abytes[dom] / t_dom / 1e9
    attn_tflops = attn_flops / (kernel_us["tree_attn_fwd"] * 1e-6) / 1e12
    kernels = {}
    for n in names:
        entry = {"us": round(kernel_us[n], 3), "entry_us": round(entry_us[n], 3)}
        if n in abytes:
            gbs = abytes[n] / (kernel_us[n] * 1e-6) / 1e9 if kernel_us[n] > 0 else 0.0
            entry.update({"algorithmic_bytes": abytes[n], "gbs": round(gbs, 1),
                          "frac_of_hbm_peak": round(gbs / peak, 4)})
        if n == "tree_attn_fwd":
            entry.update({"algorithmic_flops": attn_flops, "tflops": round(attn_tflops, 1),
                          "frac_of_tensor_peak": round(attn_tflops / tc_peak, 4),
                          "bound": "tensor" if attn_tensor else "hbm",
                          "launches": attn_launches,
                          "plan": tsd.tree_attn_plan(B, N, Hq, Hkv, D, max_slots)})
        kernels[n] = entry
    launches = launches_per_step * steps
    if tensor_bound:
        roofline = {"bound": "tensor", "kernel": dom, "achieved": round(attn_tflops, 1),
                    "peak": tc_peak, "unit": "TFLOP/s", "frac": round(attn_tflops / tc_peak, 4),
                    "traffic": ncu_traffic(dom, name), "peak_source": tc_src,
                    "algorithmic_flops_per_launch": attn_flops,
                    "algorithmic_bytes_per_launch": abytes[dom],
                    "hbm_frac": round(achieved / peak, 4)}
    else:
        roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4),
                    "traffic": ncu_traffic(dom, name), "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": abytes[dom],
                    "algorithmic_flops_per_launch": attn_flops if dom == "tree_attn_fwd" else None,
                    "tensor_frac": (round(attn_tflops / tc_peak, 4)
                                    if dom == "tree_attn_fwd" else None)}
    roofline["time_basis"] = ("kernel-only device time: CUDA events around graph replays of "
                              "[L2 flush, entry point] minus [L2 flush] alone, %d reps" % reps)
    result = {
        "metric": METRIC,
        "value": round(whole_job_rate(ms_per_step, world), 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16 (attention, fp32 accumulate); f32 (%s); int32 (tree, paths)" % (
            "rejection sampling" if stochastic else "logits argmax"),
        "data": "synthetic (seeded; shapes and distributions of the named workload)",
        "config": {"workload": desc, "name": name, "verify": verify,
                   "global_batch": B * world,
                   "seq_len": max_slots, "parallelism": "replicas (dp%d)" % world,
                   "l2": "flushed between timed steps: 256 MiB write then 256 MiB read of another "
                         "buffer, outside the timed events (cold, clean L2)",
                   "timing": "CUDA events on the launching stream around CUDA-graph replays of "
                             "the whole step (value) and of each entry point (kernels)"},
        "hbm_gbs_step": round(step_bytes / (ms_per_step * 1e-3) / 1e9, 1),
        "step_kernel_us": round(step_kernel_us, 3),
        "kernels": kernels,
        "roofline": roofline,
        "attention_tflops": round(attn_tflops, 1),
        "gpu_launches": launches,
        "wall_s_timed_region": round(t_wall, 4),
        "kernel_sum_us": round(sum(kernel_us[n] for n in step_names), 3),
        "step_calls": step_names,
        "mean_accept_len": float(A.float().mean().item()),
        "verify": (verify if not stochastic else
                   {"mode": "stochastic", "internal_rows": internal_rows,
                    "rows_with_rejection": rejected_rows, "leaf_draws": leaf_draws,
                    "plan": tsd.tree_verify_stochastic_plan(B, N, V)}),
    }
    if full:
        result["e2e"] = e2e
        result["clocks"] = clocks
        result["commit_layer_stacked"] = {
            "layers": n_layers, "us": round(stacked_us, 3),
            "algorithmic_bytes": abytes["kv_commit_path"] * n_layers,
            "gbs": round(abytes["kv_commit_path"] * n_layers / (stacked_us * 1e-6) / 1e9, 1),
            "frac_of_hbm_peak": round(abytes["kv_commit_path"] * n_layers
                                      / (stacked_us * 1e-6) / 1e9 / peak, 4)}
    return result


def config_summary(r):
    """The compact per-configuration record carried beside the headline."""
    a = r["kernels"]["tree_attn_fwd"]
    return {"workload": r["config"]["workload"], "steps_per_s": r["value"],
            "ms_per_step": r["ms_per_step"], "step_kernel_us": r["step_kernel_us"],
            "kernels_us": {n: k["us"] for n, k in r["kernels"].items()},
            "entry_us": {n: k["entry_us"] for n, k in r["kernels"].items()},
            "attention": {"bound": a["bound"], "gbs": a["gbs"],
                          "frac_of_hbm_peak": a["frac_of_hbm_peak"], "tflops": a["tflops"],
                          "frac_of_tensor_peak": a["frac_of_tensor_peak"],
                          "frac_of_binding_roof": (a["frac_of_tensor_peak"]
                                                   if a["bound"] == "tensor"
                                                   else a["frac_of_hbm_peak"]),
                          "launches": a["launches"], "plan": a["plan"]},
            "verify_frac_of_hbm_peak": r["kernels"]["tree_verify_greedy"]["frac_of_hbm_peak"]
            if "tree_verify_greedy" in r["kernels"] else None,
            "roofline": {k: r["roofline"][k] for k in ("bound", "kernel", "achieved", "unit",
                                                       "frac")},
            "steps": r["steps"], "mean_accept_len": r["mean_accept_len"]}


def gpu_arm(args, rank, world):
    import torch

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    flush = torch.empty((FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones((FLUSH_BYTES // 8,), dtype=torch.int64, device=dev)

    def flush_l2():
        # write one buffer larger than L2, then read another: the timed step
        # starts with a cold L2 holding clean lines, so no write-back of the
        # flush's dirty lines is charged to the kernels
        flush.zero_()
        flush_rd.sum()

    res = measure_workload(args.workload, args, rank, world, dev, flush_l2, full=True,
                           verify=args.verify)
    if world == 1 and args.configs and args.verify == "greedy":
        sub = argparse.Namespace(**vars(args))
        sub.steps = max(3, min(args.steps, args.config_steps))
        sub.batch = None
        others = {}
        for name in CONFIG_SET:
            if name == args.workload:
                continue
            r = measure_workload(name, sub, rank, 1, dev, flush_l2, full=False)
            others[name] = config_summary(r)
            torch.cuda.empty_cache()
        res["configs"] = others
    return res


def budget_arm(args, rank, world):
    """BASTION's online tree budget on its own workload (B=8 marginals over
    16 positions, verify on the 8B-shaped layer with prefix 2048): the verify
    step (a1-a4) is timed at N = 16..256, a roofline cost model is calibrated
    on those times, and the budgeted step runs best-first construction at 256
    nodes, the device-side choice of each sequence's size, and a1-a4 on the
    chosen prefixes of the trees, all on one stream."""
    import torch
    import torch.distributed as dist

    import tree_speculative_decoding_virtual_gb300 as tsd

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    hbm, hbm_src, _ = load_peaks()
    tc, tc_src = load_tensor_peak()
    q_m, root = gen.bastion_marginals()
    c = gen.BASTION
    qd, rootd = torch.from_numpy(q_m).to(dev), torch.from_numpy(root).to(dev)
    flush = torch.empty((FLUSH_BYTES,), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones((FLUSH_BYTES // 8,), dtype=torch.int64, device=dev)

    def flush_l2():
        flush.zero_()
        flush_rd.sum()

    def capture(fn):
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            fn()
        torch.cuda.current_stream().wait_stream(side)
        with torch.cuda.graph(g):
            fn()
        return g

    def timed(g, reps):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(reps)]
        for a_, b_ in ev:
            flush_l2()
            a_.record(stream)
            g.replay()
            b_.record(stream)
        torch.cuda.synchronize()
        return 1000.0 * sum(a_.elapsed_time(b_) for a_, b_ in ev) / reps

    def verify_setup(N):
        """Best-first tree of N nodes on the GPU, the verify inputs built on it,
        and the a1-a4 calls on device buffers."""
        bf_ws = torch.empty(tsd.best_first_workspace_bytes(*q_m.shape, N), dtype=torch.uint8,
                            device=dev)
        outs = [torch.empty((c["B"], N), dtype=torch.int32, device=dev) for _ in range(3)]
        rho = torch.empty((c["B"], N), dtype=torch.float32, device=dev)
        ahat = torch.empty((c["B"],), dtype=torch.float64, device=dev)
        bf = lambda: tsd.best_first_tree_build(qd, rootd, N, *outs, rho, ahat, workspace=bf_ws)
        bf()
        torch.cuda.synchronize()
        par_h, tok_h, dep_h = [x.cpu().numpy() for x in outs]
        top1 = np.argmax(q_m, axis=-1)  # input synthesis only: plants target choices
        inp = gen.bastion_verify_inputs(par_h, tok_h, dep_h, top1)
        T = lambda a, dt=None: (torch.from_numpy(np.ascontiguousarray(a)).view(dt)
                                if dt is not None else torch.from_numpy(np.ascontiguousarray(a))).to(dev)
        Bq, Nq, Hq, Hkv, D, V, Dm = inp.B, inp.N_max, inp.Hq, inp.Hkv, inp.D, inp.V, inp.D_max
        d = dict(parent=T(inp.parent), n_nodes=T(inp.n_nodes), prefix=T(inp.prefix_len),
                 tokens=T(inp.tokens), logits=T(inp.logits), q=T(inp.q, torch.bfloat16),
                 table=T(inp.cache.block_table), kc=T(inp.cache.k, torch.bfloat16),
                 vc=T(inp.cache.v, torch.bfloat16))
        max_slots = int((inp.prefix_len + N).max())
        W = (Nq + 31) // 32
        i32 = dict(dtype=torch.int32, device=dev)
        anc = torch.empty((Bq, Nq + 1, Dm + 1), **i32)
        depth = torch.empty((Bq, Nq), **i32)
        mask = torch.empty((Bq, Nq, W), **i32)
        err = torch.empty((Bq,), **i32)
        out = torch.empty((Bq, Nq, Hq, D), dtype=torch.bfloat16, device=dev)
        attn_ws = torch.empty((tsd.tree_attn_workspace_bytes(Bq, Nq, Hq, Hkv, D, max_slots),),
                              dtype=torch.uint8, device=dev)
        ver_ws = torch.zeros((tsd.tree_verify_workspace_bytes(Bq, Nq, V),), dtype=torch.uint8,
                             device=dev)
        am = torch.empty((Bq, Nq), **i32)
        A = torch.empty((Bq,), **i32)
        leaf = torch.empty((Bq,), **i32)
        path = torch.empty((Bq, Dm + 1), **i32)
        bonus = torch.empty((Bq,), **i32)
        new_len = torch.empty((Bq,), **i32)
        moved = torch.empty((Bq,), **i32)
        status = torch.zeros((1,), **i32)

        def verify(n_nodes=None):
            nn_ = d["n_nodes"] if n_nodes is None else n_nodes
            tsd.tree_build_ancestors(d["parent"], nn_, Dm, anc, depth, mask, err)
            tsd.tree_attn_fwd(d["q"], d["kc"], d["vc"], d["table"], d["prefix"], nn_, mask, err,
                              max_slots, out=out, workspace=attn_ws, status=status)
            tsd.tree_verify_greedy(d["logits"], d["tokens"], d["parent"], anc, depth, mask, nn_,
                                   err, Dm, am, A, leaf, path, bonus, workspace=ver_ws)
            tsd.kv_commit_path(d["kc"], d["vc"], d["table"], d["prefix"], nn_, A, path, err, Nq,
                               Dm, new_len=new_len, moved=moved, status=status)
        return inp, bf, rho, verify, status

    reps = max(3, min(args.steps, 100))
    Ns = [16, 32, 64, 128, 256]
    t_verify, t_roof, t_bf = {}, {}, {}
    keep = None
    for N in Ns:
        inp, bf, rho, verify, status = verify_setup(N)
        for _ in range(args.warmup):
            verify()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        t_verify[N] = timed(capture(verify), reps)
        t_bf[N] = timed(capture(bf), reps)
        t_roof[N] = tsd.verify_step_cost(inp.B, inp.Hq, inp.Hkv, inp.D, inp.prefix_len, inp.V,
                                         inp.D_max, N, hbm, tc)[2]
        if N == Ns[-1]:
            keep = (inp, bf, rho, verify, status)
    alpha, beta = tsd.budget_calibrate([t_roof[N] for N in Ns], [t_verify[N] for N in Ns])
    inp, bf, rho, verify, status = keep
    n_max = Ns[-1]
    roof_of = lambda n: tsd.verify_step_cost(inp.B, inp.Hq, inp.Hkv, inp.D, inp.prefix_len, inp.V,
                                             min(16, max(n - 1, 0)), n, hbm, tc)[2]
    t_draft = t_bf[n_max]          # the tree construction; the drafter's own pass is not modelled
    l_ar = alpha * roof_of(1) + beta  # a 1-node tree is a plain decode step
    cost_h = np.array([t_draft + alpha * roof_of(max(n, 1)) + beta for n in range(n_max + 1)])
    cost = torch.from_numpy(cost_h.astype(np.float32)).to(dev)
    n_opt = torch.empty((inp.B,), dtype=torch.int32, device=dev)
    s_opt = torch.empty((inp.B,), dtype=torch.float32, device=dev)

    def budgeted_step():
        bf()
        tsd.budget_select(rho, cost, l_ar, n_opt, s_opt)
        verify(n_opt)

    for _ in range(args.warmup):
        budgeted_step()
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    g_step = capture(budgeted_step)
    g_sel = capture(lambda: tsd.budget_select(rho, cost, l_ar, n_opt, s_opt))
    sampler = ClockSampler(local) if rank == 0 else None
    if world > 1:
        dist.barrier()
    ms = max_over_ranks(timed(g_step, args.steps) / 1000.0, world, dev)
    clocks = sampler.stop() if sampler else None
    sel_us = timed(g_sel, reps)
    n_h = n_opt.cpu().numpy()
    if rank != 0:
        return None
    model = {N: alpha * t_roof[N] + beta for N in Ns}
    step_bytes = sum(tsd.verify_step_cost(1, inp.Hq, inp.Hkv, inp.D, [int(inp.prefix_len[b])],
                                          inp.V, inp.D_max, int(n_h[b]), hbm, tc)[0]
                     for b in range(inp.B)) + 4.0 * q_m.size
    return {
        "metric": METRIC,
        "value": round(whole_job_rate(ms, world), 2),
        "unit": "steps/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp32 marginals, path scores and budget choice; bf16 attention; f32 logits",
        "data": "synthetic (seeded; shapes and distributions of the named workload)",
        "config": {"workload": "BASTION-style budgeted step: B=8, K=16, V=32000 marginals, "
                               "best-first at 256 nodes, online size choice, verify on Hq=32, "
                               "Hkv=8, D=128, prefix 2048", "name": "bastion-budget",
                   "global_batch": inp.B * world, "parallelism": "replicas (dp%d)" % world,
                   "l2": "flushed between timed steps (256 MiB write, 256 MiB read)"},
        "budget": {"N": Ns, "t_verify_us": [round(t_verify[N], 3) for N in Ns],
                   "t_roofline_us": [round(t_roof[N], 3) for N in Ns],
                   "t_model_us": [round(model[N], 3) for N in Ns],
                   "alpha": alpha, "beta_us": beta, "t_draft_us": round(t_draft, 3),
                   "l_ar_us": round(l_ar, 3), "n_opt": n_h.tolist(),
                   "s_opt": [round(float(x), 4) for x in s_opt.cpu().numpy()],
                   "select_us": round(sel_us, 3),
                   "peaks": {"hbm_gbs": hbm, "hbm_source": hbm_src, "bf16_tflops": tc,
                             "tensor_source": tc_src}},
        "roofline": {"bound": "hbm", "kernel": "whole budgeted step",
                     "achieved": round(step_bytes / (ms * 1e-3) / 1e9, 1), "peak": hbm,
                     "unit": "GB/s", "frac": round(step_bytes / (ms * 1e-3) / 1e9 / hbm, 4),
                     "traffic": None, "peak_source": hbm_src},
        "gpu_launches": 8 * args.steps,
        "clocks": clocks,
    }


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="70b",
                    help="headline workload (default: the long-context 70B-shaped layer, the "
                         "largest configuration on one GPU)")
    ap.add_argument("--verify", default="greedy", choices=["greedy", "stochastic"],
                    help="a3: greedy (argmax) or stochastic (modified rejection sampling)")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the other configurations measured beside the headline")
    ap.add_argument("--config-steps", type=int, default=2000,
                    help="timed steps for each of the other configurations")
    ap.add_argument("--batch", type=int, default=None,
                    help="keep the first B sequences of the headline workload (profiling)")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(reference_arm(args, world)), flush=True)
        return 0

    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    base = None
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and args.verify == "greedy"
            and not args.workload.startswith("bastion") and args.workload != "dynamic"):
        base = cpu_baseline(args.workload)
    res = (budget_arm if args.workload == "bastion-budget" else gpu_arm)(args, rank, world)
    if rank == 0:
        res["cpu_baseline"] = base
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def reference_arm(args, world):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the workload (attention on a sample of rows, the rest in full),
    scaled to full-step units."""
    name = args.workload if not (args.workload.startswith("bastion")
                                 or args.workload == "dynamic") else "8b"
    threads = os.cpu_count() or 1
    frac = oracle_sample_fraction(name)
    # size the run to a few minutes at most: measure one sampled step first
    probe = run_oracle_child(name, 1, frac, threads)
    per_sample = probe["wall"]
    budget = 150.0
    steps = max(1, min(args.steps, int(budget / max(per_sample, 1e-3)) - args.warmup))
    res = run_oracle_child(name, steps, frac, threads)
    sec = res["sec_per_full_step"]
    _, desc = workload_inputs(name)
    value = 1.0 / sec
    sample = ("%d oracle steps of the %s workload (of %d requested); each runs ancestors, verify "
              "and commit in full and attention on %d of %d (seq, node, q-head) rows, scaled to "
              "the full row count" % (steps, name, args.steps, res["sample_rows"], res["total_rows"]))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup, "ms_per_step": 1000.0 * sec,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded; shapes and distributions of the named workload)",
            "config": {"workload": desc, "name": name, "global_batch": None,
                       "parallelism": "host cores"},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


if __name__ == "__main__":
    sys.exit(main())
