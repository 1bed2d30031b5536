"""The oracle: a plain, slow, CPU implementation of the tree-verify hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
executes this package; only the tests, the smoke check and the benchmark's
CPU-baseline leg (and its reference arm) do.  It shares no code with the CUDA
library and does not import it.

Sources, cited by page title and section:

* [EP-zh] "EAGLE-Pangu: Accelerator-Safe Tree Speculative Decoding on Ascend
  NPUs", technical summary (gist.science/zh/paper/2603.08088): 2.1 branchable
  KV cache, 2.2 accelerator-safe tree tensor semantics, 2.3 fused tree-masked
  teacher execution.
* [EP-pt] the same paper's Portuguese technical summary
  (gist.science/pt/paper/2603.08088), section 2 "Metodologia e Arquitetura".
* [BASTION] "Resumo Técnico: BASTION" (gist.science/pt/paper/2605.29727),
  Methodology 1 (block-diffusion drafting, path score), 2 (acceptance
  surrogate and best-first expansion) and 3 (hardware-aware online budget
  controller).
* [Blog] "Speculative Decoding Hierárquico: Medusa, EAGLE-2 e Multi-Token
  Prediction" (produtoramaxvision.com.br): sections on modified rejection
  sampling, the speed-up model and Medusa tree attention.

Floating point is fp64 except where a step is defined in fp32 on purpose (the
path score product of best-first construction, so that rankings are
reproducible bit for bit).  Every function states the readings taken where the
pages are silent.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
(closed forms, library routines, brute force, invariants, the pages' example
trees); none is "parity unpinned".
"""

from .tree import (ERR_RANGE, ERR_CYCLE, ERR_TOO_DEEP, ERR_CLOSURE, ERR_ROOT, ERR_COUNT,
                   build_ancestors, ancestor_chain)
from .attention import bf16_to_f64, tree_attention, gather_sequence_kv, physical_slots
from .verify import verify_greedy
from .commit import commit_path, commit_remap
from .best_first import best_first_tree, ranked_tokens
from .rejection import modified_rejection_step, residual_distribution
from .budget import verify_step_cost, calibrate, speedup_curve, budget_select, cost_table
from .stochastic import node_decision, tree_verify_stochastic, tree_verify_stochastic_all
from .dynamic_tree import (dynamic_tree, expand_level, new_pool, pool_base, pool_size,
                           rerank as dynamic_tree_rerank)

__all__ = [
    "ERR_RANGE", "ERR_CYCLE", "ERR_TOO_DEEP", "ERR_CLOSURE", "ERR_ROOT", "ERR_COUNT",
    "build_ancestors", "ancestor_chain", "bf16_to_f64", "tree_attention", "gather_sequence_kv",
    "verify_greedy", "commit_path", "commit_remap", "physical_slots", "best_first_tree",
    "ranked_tokens",
    "modified_rejection_step", "residual_distribution",
    "verify_step_cost", "calibrate", "speedup_curve", "budget_select", "cost_table",
    "node_decision", "tree_verify_stochastic", "tree_verify_stochastic_all",
    "dynamic_tree", "expand_level", "new_pool", "pool_base", "pool_size", "dynamic_tree_rerank",
]
