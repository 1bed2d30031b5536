"""Python binding of libtsd.so, the GB300 tree-speculative-decoding verify path.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch supplies device memory and the current stream.  Each call has the
name of its C entry point without the ``tsd_`` prefix; outputs and workspaces
may be passed in (no allocation inside the call, e.g. under CUDA-graph
capture) or are allocated here when omitted.

Importing the package loads the shared library and fails loudly if it has not
been built (``tree_speculative_decoding_virtual_gb300._build.build()``).
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

from ._build import LIB as _LIB_PATH

TSD_OK, TSD_ERR_ARG, TSD_ERR_LIMIT, TSD_ERR_WORKSPACE, TSD_ERR_CUDA = 0, -1, -2, -3, -4
_ERR_NAMES = {TSD_ERR_ARG: "TSD_ERR_ARG", TSD_ERR_LIMIT: "TSD_ERR_LIMIT",
              TSD_ERR_WORKSPACE: "TSD_ERR_WORKSPACE", TSD_ERR_CUDA: "TSD_ERR_CUDA"}

TREE_RANGE, TREE_CYCLE, TREE_TOO_DEEP, TREE_CLOSURE, TREE_ROOT, TREE_COUNT = 1, 2, 4, 8, 16, 32
STATUS_BAD_PAGE, STATUS_BAD_LEN, STATUS_BAD_PATH, STATUS_TIMEOUT = 1, 2, 4, 8
OPT_WAIT_LIMIT_NS, OPT_TEST_STALL = 0, 1

# C signatures: (name, restype, argtypes)
_P, _I, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_D = ctypes.c_double
SIGNATURES = {
    "tsd_version": (ctypes.c_char_p, []),
    "tsd_set_option": (_I, [_I, _I64]),
    "tsd_get_option": (_I64, [_I]),
    "tsd_tree_build_ancestors": (_I, [_P, _P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tsd_tree_attn_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "tsd_tree_attn_launches": (_I, [_I, _I, _I, _I, _I, _I]),
    "tsd_tree_attn_plan": (_I, [_I, _I, _I, _I, _I, _I, _P]),
    "tsd_tree_attn_fwd": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F,
                               _P, _P, _P, _SZ, _P, _P]),
    "tsd_tree_attn_fwd_remap": (_I, [_P, _P, _P, _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                     _F, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "tsd_tree_verify_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tsd_tree_verify_greedy": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                    _P, _P, _SZ, _P]),
    "tsd_tree_verify_greedy_commit": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P,
                                           _P, _P, _P, _P, _SZ, _P, _P, _I, _I64, _P, _I, _I, _P,
                                           _I, _I, _P, _P, _P, _P]),
    "tsd_tree_verify_static_capacity": (_SZ, []),
    "tsd_tree_verify_greedy_static": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P,
                                           _P, _P, _P, _P]),
    "tsd_tree_verify_stochastic_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tsd_tree_verify_stochastic": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P,
                                        _P, _P, _P, _P, _SZ, _P, _P]),
    "tsd_tree_verify_stochastic_plan": (_I, [_I, _I, _I, _P, _P]),
    "tsd_kv_commit_path": (_I, [_P, _P, _I, _I64, _P, _I, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                _I, _P, _P, _P, _P]),
    "tsd_kv_commit_path_from": (_I, [_P, _P, _I, _I64, _P, _I, _I, _P, _P, _P, _P, _P, _P, _I, _I,
                                     _I, _I, _I, _P, _P, _P, _P]),
    "tsd_kv_commit_remap": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "tsd_best_first_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "tsd_best_first_tree_build": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "tsd_dynamic_tree_workspace_bytes": (_SZ, [_I, _I, _I]),
    "tsd_dynamic_tree_expand": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _I, _P, _P,
                                     _SZ, _P]),
    "tsd_dynamic_tree_rerank": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "tsd_verify_step_cost": (_I, [_I, _I, _I, _I, _P, _I, _I, _I, _D, _D, _P, _P, _P]),
    "tsd_budget_calibrate": (_I, [_P, _P, _I, _P, _P]),
    "tsd_budget_select": (_I, [_P, _I, _I, _P, _F, _P, _P, _P]),
}


class TsdError(RuntimeError):
    pass


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError("libtsd.so is not built at %s; run "
                          "tree_speculative_decoding_virtual_gb300._build.build()" % _LIB_PATH)
    lib = ctypes.CDLL(_LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
LIB_PATH = _LIB_PATH


def _check(rc: int, what: str):
    if rc != TSD_OK:
        raise TsdError("%s failed: %s" % (what, _ERR_NAMES.get(rc, rc)))


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise TsdError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise TsdError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TsdError("%s must be %s, got %s" % (name, dtype, t.dtype))
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


# ---------------------------------------------------------------------------
# a1
# ---------------------------------------------------------------------------

def tree_build_ancestors(parent, n_nodes, D_max, anc=None, depth=None, mask=None, err=None,
                         stream=None):
    """parent int32 [B][N_max]; n_nodes int32 [B] or None.  Returns
    (anc [B][N_max+1][D_max+1], depth [B][N_max], mask uint32-as-int32
    [B][N_max][W], err [B])."""
    B, N_max = parent.shape
    W = (N_max + 31) // 32
    anc = anc if anc is not None else _empty((B, N_max + 1, D_max + 1), torch.int32, parent)
    depth = depth if depth is not None else _empty((B, N_max), torch.int32, parent)
    mask = mask if mask is not None else _empty((B, N_max, W), torch.int32, parent)
    err = err if err is not None else _empty((B,), torch.int32, parent)
    rc = lib.tsd_tree_build_ancestors(_ptr(parent, torch.int32, "parent"),
                                      _ptr(n_nodes, torch.int32, "n_nodes"), B, N_max, D_max,
                                      _ptr(anc, torch.int32, "anc"), _ptr(depth, torch.int32, "depth"),
                                      _ptr(mask, torch.int32, "mask"), _ptr(err, torch.int32, "err"),
                                      _stream(stream))
    _check(rc, "tree_build_ancestors")
    return anc, depth, mask, err


# ---------------------------------------------------------------------------
# a2
# ---------------------------------------------------------------------------

def tree_attn_workspace_bytes(B, N_max, Hq, Hkv, D, max_slots) -> int:
    return int(lib.tsd_tree_attn_workspace_bytes(B, N_max, Hq, Hkv, D, max_slots))


def tree_attn_launches(B, N_max, Hq, Hkv, D, max_slots) -> int:
    """Kernels one tree_attn_fwd call launches for these sizes."""
    return int(lib.tsd_tree_attn_launches(B, N_max, Hq, Hkv, D, max_slots))


def tree_attn_plan(B, N_max, Hq, Hkv, D, max_slots) -> dict:
    """The launch shape tree_attn_fwd picks for these sizes on this device."""
    info = (ctypes.c_int32 * 8)()
    _check(lib.tsd_tree_attn_plan(B, N_max, Hq, Hkv, D, max_slots, info), "tree_attn_plan")
    keys = ["mode", "two_blocks_per_sm", "rows_per_block", "row_blocks", "splits", "keys_per_split",
            "grid_blocks", "direct"]
    return dict(zip(keys, [int(x) for x in info]))


def tree_attn_fwd(q, k_cache, v_cache, block_table, prefix_len, n_nodes, mask, err, max_slots,
                  scale=None, out=None, lse=None, want_lse=True, workspace=None, status=None,
                  stream=None, remap=None):
    """q bf16 [B][N_max][Hq][D]; caches bf16 [num_blocks][Hkv][16][D];
    block_table int32 [B][max_blocks].  remap: None, or (remap_src [B][D_max+1],
    remap_base [B], remap_len [B], tail_base [B]) from kv_commit_remap, to read
    the committed sequence through a deferred commit.  Returns (out bf16
    [B][N_max][Hq][D], lse float32 [B][N_max][Hq] or None)."""
    B, N_max, Hq, D = q.shape
    num_blocks, Hkv = k_cache.shape[0], k_cache.shape[1]
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / float(D) ** 0.5
    out = out if out is not None else _empty(q.shape, torch.bfloat16, q)
    if lse is None and want_lse:
        lse = _empty((B, N_max, Hq), torch.float32, q)
    need = tree_attn_workspace_bytes(B, N_max, Hq, Hkv, D, max_slots)
    if workspace is None and need > 0:
        workspace = _empty((need,), torch.uint8, q)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if remap is not None:
        src, rbase, rlen, tbase = remap
        rc = lib.tsd_tree_attn_fwd_remap(
            _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k_cache"),
            _ptr(v_cache, torch.bfloat16, "v_cache"),
            _ptr(block_table, torch.int32, "block_table"), max_blocks, num_blocks,
            _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(n_nodes, torch.int32, "n_nodes"),
            _ptr(mask, torch.int32, "mask"), _ptr(err, torch.int32, "err"), B, N_max, Hq, Hkv, D,
            int(max_slots), float(scale), _ptr(src, torch.int32, "remap_src"),
            int(src.shape[1]) if src is not None else 0, _ptr(rbase, torch.int32, "remap_base"),
            _ptr(rlen, torch.int32, "remap_len"), _ptr(tbase, torch.int32, "tail_base"),
            _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
            _ptr(workspace, None, "workspace"), ws_bytes, _ptr(status, torch.int32, "status"),
            _stream(stream))
        _check(rc, "tree_attn_fwd_remap")
        return out, lse
    rc = lib.tsd_tree_attn_fwd(
        _ptr(q, torch.bfloat16, "q"), _ptr(k_cache, torch.bfloat16, "k_cache"),
        _ptr(v_cache, torch.bfloat16, "v_cache"), _ptr(block_table, torch.int32, "block_table"),
        max_blocks, num_blocks, _ptr(prefix_len, torch.int32, "prefix_len"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(mask, torch.int32, "mask"),
        _ptr(err, torch.int32, "err"), B, N_max, Hq, Hkv, D, int(max_slots), float(scale),
        _ptr(out, torch.bfloat16, "out"), _ptr(lse, torch.float32, "lse"),
        _ptr(workspace, None, "workspace"), ws_bytes,
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "tree_attn_fwd")
    return out, lse


# ---------------------------------------------------------------------------
# a3
# ---------------------------------------------------------------------------

def tree_verify_workspace_bytes(B, N_max, V) -> int:
    return int(lib.tsd_tree_verify_workspace_bytes(B, N_max, V))


def tree_verify_greedy(logits, tokens, parent, anc, depth, mask, n_nodes, err, D_max,
                       argmax=None, accept_len=None, leaf=None, path=None, bonus=None,
                       workspace=None, stream=None):
    """logits float32 [B][N_max][V].  Returns (argmax [B][N_max], accept_len
    [B], leaf [B], path [B][D_max+1], bonus [B]).  A workspace passed in must
    be zero-filled before its first use (the call leaves it zero-filled)."""
    B, N_max, V = logits.shape
    argmax = argmax if argmax is not None else _empty((B, N_max), torch.int32, logits)
    accept_len = accept_len if accept_len is not None else _empty((B,), torch.int32, logits)
    leaf = leaf if leaf is not None else _empty((B,), torch.int32, logits)
    path = path if path is not None else _empty((B, D_max + 1), torch.int32, logits)
    bonus = bonus if bonus is not None else _empty((B,), torch.int32, logits)
    need = tree_verify_workspace_bytes(B, N_max, V)
    if workspace is None:
        workspace = torch.zeros((max(need, 1),), dtype=torch.uint8, device=logits.device)
    rc = lib.tsd_tree_verify_greedy(
        _ptr(logits, torch.float32, "logits"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(parent, torch.int32, "parent"), _ptr(anc, torch.int32, "anc"),
        _ptr(depth, torch.int32, "depth"), _ptr(mask, torch.int32, "mask"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(err, torch.int32, "err"), B, N_max, V, D_max,
        _ptr(argmax, torch.int32, "argmax"), _ptr(accept_len, torch.int32, "accept_len"),
        _ptr(leaf, torch.int32, "leaf"), _ptr(path, torch.int32, "path"),
        _ptr(bonus, torch.int32, "bonus"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "tree_verify_greedy")
    return argmax, accept_len, leaf, path, bonus


def tree_verify_greedy_commit(logits, tokens, parent, anc, depth, mask, n_nodes, err, D_max,
                              k_cache, v_cache, block_table, prefix_len, num_layers=1,
                              argmax=None, accept_len=None, leaf=None, path=None, bonus=None,
                              new_len=None, moved=None, status=None, workspace=None, stream=None):
    """tree_verify_greedy, then, in the same launch, kv_commit_path of the
    accepted paths (caches as kv_commit_path takes them).  Returns (argmax,
    accept_len, leaf, path, bonus, new_len, moved)."""
    B, N_max, V = logits.shape
    if k_cache.dim() == 5:
        num_layers = k_cache.shape[0]
        num_blocks, Hkv, _, D = k_cache.shape[1:]
        layer_stride = k_cache.stride(0)
    else:
        num_blocks, Hkv, _, D = k_cache.shape
        layer_stride = k_cache.numel()
    max_blocks = block_table.shape[1]
    argmax = argmax if argmax is not None else _empty((B, N_max), torch.int32, logits)
    accept_len = accept_len if accept_len is not None else _empty((B,), torch.int32, logits)
    leaf = leaf if leaf is not None else _empty((B,), torch.int32, logits)
    path = path if path is not None else _empty((B, D_max + 1), torch.int32, logits)
    bonus = bonus if bonus is not None else _empty((B,), torch.int32, logits)
    new_len = new_len if new_len is not None else _empty((B,), torch.int32, logits)
    moved = moved if moved is not None else _empty((B,), torch.int32, logits)
    need = tree_verify_workspace_bytes(B, N_max, V)
    if workspace is None:
        workspace = torch.zeros((max(need, 1),), dtype=torch.uint8, device=logits.device)
    rc = lib.tsd_tree_verify_greedy_commit(
        _ptr(logits, torch.float32, "logits"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(parent, torch.int32, "parent"), _ptr(anc, torch.int32, "anc"),
        _ptr(depth, torch.int32, "depth"), _ptr(mask, torch.int32, "mask"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(err, torch.int32, "err"), B, N_max, V, D_max,
        _ptr(argmax, torch.int32, "argmax"), _ptr(accept_len, torch.int32, "accept_len"),
        _ptr(leaf, torch.int32, "leaf"), _ptr(path, torch.int32, "path"),
        _ptr(bonus, torch.int32, "bonus"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(),
        _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        num_layers, layer_stride, _ptr(block_table, torch.int32, "block_table"), max_blocks,
        num_blocks, _ptr(prefix_len, torch.int32, "prefix_len"), Hkv, D,
        _ptr(new_len, torch.int32, "new_len"), _ptr(moved, torch.int32, "moved"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "tree_verify_greedy_commit")
    return argmax, accept_len, leaf, path, bonus, new_len, moved


def tree_verify_static_capacity() -> int:
    return int(lib.tsd_tree_verify_static_capacity())


def tree_verify_greedy_static(logits, tokens, parent, anc, depth, mask, n_nodes, err, D_max,
                              argmax=None, accept_len=None, leaf=None, path=None, bonus=None,
                              stream=None):
    """tree_verify_greedy without a workspace, for callers that cannot
    allocate device memory: the library's fixed device array serves as
    scratch (calls that overlap on the GPU race on it).  Outputs passed in
    are written in place; omitted ones are allocated here."""
    B, N_max, V = logits.shape
    argmax = argmax if argmax is not None else _empty((B, N_max), torch.int32, logits)
    accept_len = accept_len if accept_len is not None else _empty((B,), torch.int32, logits)
    leaf = leaf if leaf is not None else _empty((B,), torch.int32, logits)
    path = path if path is not None else _empty((B, D_max + 1), torch.int32, logits)
    bonus = bonus if bonus is not None else _empty((B,), torch.int32, logits)
    rc = lib.tsd_tree_verify_greedy_static(
        _ptr(logits, torch.float32, "logits"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(parent, torch.int32, "parent"), _ptr(anc, torch.int32, "anc"),
        _ptr(depth, torch.int32, "depth"), _ptr(mask, torch.int32, "mask"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(err, torch.int32, "err"), B, N_max, V, D_max,
        _ptr(argmax, torch.int32, "argmax"), _ptr(accept_len, torch.int32, "accept_len"),
        _ptr(leaf, torch.int32, "leaf"), _ptr(path, torch.int32, "path"),
        _ptr(bonus, torch.int32, "bonus"), _stream(stream))
    _check(rc, "tree_verify_greedy_static")
    return argmax, accept_len, leaf, path, bonus


def tree_verify_stochastic_workspace_bytes(B: int, N_max: int, V: int) -> int:
    return int(lib.tsd_tree_verify_stochastic_workspace_bytes(B, N_max, V))


def tree_verify_stochastic(logits, q_draft, tokens, parent, n_nodes, err, u_accept, u_draw, D_max,
                           next=None, draw=None, accept_len=None, leaf=None, path=None,
                           bonus=None, workspace=None, status=None, stream=None):
    """Modified rejection sampling over the tree.  logits, q_draft float32
    [B][N_max][V]; u_accept, u_draw float32 [B][N_max] uniforms; err from
    tree_build_ancestors (required).  Returns (next [B][N_max], draw
    [B][N_max], accept_len [B], leaf [B], path [B][D_max+1], bonus [B]).  A
    workspace passed in must have its first 4*B bytes (the tickets) zeroed
    before its first use; calls leave them zeroed."""
    B, N_max, V = logits.shape
    next = next if next is not None else _empty((B, N_max), torch.int32, logits)
    draw = draw if draw is not None else _empty((B, N_max), torch.int32, logits)
    accept_len = accept_len if accept_len is not None else _empty((B,), torch.int32, logits)
    leaf = leaf if leaf is not None else _empty((B,), torch.int32, logits)
    path = path if path is not None else _empty((B, D_max + 1), torch.int32, logits)
    bonus = bonus if bonus is not None else _empty((B,), torch.int32, logits)
    need = tree_verify_stochastic_workspace_bytes(B, N_max, V)
    if workspace is None:
        workspace = torch.zeros((max(need, 1),), dtype=torch.uint8, device=logits.device)
    if tuple(q_draft.shape) != (B, N_max, V):
        raise TsdError("q_draft must have the shape of logits")
    rc = lib.tsd_tree_verify_stochastic(
        _ptr(logits, torch.float32, "logits"), _ptr(q_draft, torch.float32, "q_draft"),
        _ptr(tokens, torch.int32, "tokens"), _ptr(parent, torch.int32, "parent"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(err, torch.int32, "err"),
        _ptr(u_accept, torch.float32, "u_accept"), _ptr(u_draw, torch.float32, "u_draw"),
        B, N_max, V, D_max, _ptr(next, torch.int32, "next"), _ptr(draw, torch.int32, "draw"),
        _ptr(accept_len, torch.int32, "accept_len"), _ptr(leaf, torch.int32, "leaf"),
        _ptr(path, torch.int32, "path"), _ptr(bonus, torch.int32, "bonus"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "tree_verify_stochastic")
    return next, draw, accept_len, leaf, path, bonus


def tree_verify_stochastic_plan(B: int, N_max: int, V: int):
    """(CTAs per node, floats of the row per CTA) the call picks on the
    current device."""
    c, s = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib.tsd_tree_verify_stochastic_plan(B, N_max, V, ctypes.byref(c), ctypes.byref(s)),
           "tree_verify_stochastic_plan")
    return c.value, s.value


# ---------------------------------------------------------------------------
# a4
# ---------------------------------------------------------------------------

def kv_commit_path(k_cache, v_cache, block_table, prefix_len, n_nodes, accept_len, path, err,
                   N_max, D_max, num_layers=1, new_len=None, moved=None, status=None,
                   stream=None, tail_base=None):
    """Caches bf16 [num_layers][num_blocks][Hkv][16][D] (or without the layer
    axis).  Commits in place; tail_base int32 [B]: the tree sits there instead
    of right after the prefix.  Returns (new_len [B], moved [B])."""
    if k_cache.dim() == 5:
        num_layers = k_cache.shape[0]
        num_blocks, Hkv, _, D = k_cache.shape[1:]
        layer_stride = k_cache.stride(0)
    else:
        num_blocks, Hkv, _, D = k_cache.shape
        layer_stride = k_cache.numel()
    B, max_blocks = block_table.shape
    new_len = new_len if new_len is not None else _empty((B,), torch.int32, k_cache)
    moved = moved if moved is not None else _empty((B,), torch.int32, k_cache)
    if tail_base is not None:
        rc = lib.tsd_kv_commit_path_from(
            _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
            num_layers, layer_stride, _ptr(block_table, torch.int32, "block_table"), max_blocks,
            num_blocks, _ptr(prefix_len, torch.int32, "prefix_len"),
            _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(accept_len, torch.int32, "accept_len"),
            _ptr(path, torch.int32, "path"), _ptr(err, torch.int32, "err"),
            _ptr(tail_base, torch.int32, "tail_base"), B, N_max, Hkv, D, D_max,
            _ptr(new_len, torch.int32, "new_len"), _ptr(moved, torch.int32, "moved"),
            _ptr(status, torch.int32, "status"), _stream(stream))
        _check(rc, "kv_commit_path_from")
        return new_len, moved
    rc = lib.tsd_kv_commit_path(
        _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        num_layers, layer_stride, _ptr(block_table, torch.int32, "block_table"), max_blocks,
        num_blocks, _ptr(prefix_len, torch.int32, "prefix_len"),
        _ptr(n_nodes, torch.int32, "n_nodes"), _ptr(accept_len, torch.int32, "accept_len"),
        _ptr(path, torch.int32, "path"), _ptr(err, torch.int32, "err"), B, N_max, Hkv, D, D_max,
        _ptr(new_len, torch.int32, "new_len"), _ptr(moved, torch.int32, "moved"),
        _ptr(status, torch.int32, "status"), _stream(stream))
    _check(rc, "kv_commit_path")
    return new_len, moved


def kv_commit_remap(prefix_len, n_nodes, accept_len, path, err, N_max, D_max, tail_base=None,
                    status=None, stream=None):
    """Deferred commit: records where each committed entry is, moves nothing.
    Returns (remap_src [B][D_max+1], remap_base [B], remap_len [B], new_len [B],
    next_tail [B]); pass (remap_src, remap_base, remap_len, next_tail) as
    tree_attn_fwd(remap=...) in the next step, with the next tree's K/V
    written from next_tail on."""
    B = prefix_len.shape[0]
    outs = [_empty((B, D_max + 1), torch.int32, prefix_len)] + [
        _empty((B,), torch.int32, prefix_len) for _ in range(4)]
    rc = lib.tsd_kv_commit_remap(
        _ptr(prefix_len, torch.int32, "prefix_len"), _ptr(n_nodes, torch.int32, "n_nodes"),
        _ptr(accept_len, torch.int32, "accept_len"), _ptr(path, torch.int32, "path"),
        _ptr(err, torch.int32, "err"), _ptr(tail_base, torch.int32, "tail_base"), B, N_max, D_max,
        *[_ptr(o, torch.int32, "out") for o in outs], _ptr(status, torch.int32, "status"),
        _stream(stream))
    _check(rc, "kv_commit_remap")
    return tuple(outs)


# ---------------------------------------------------------------------------
# a5
# ---------------------------------------------------------------------------

def best_first_workspace_bytes(B, K, V, N) -> int:
    return int(lib.tsd_best_first_workspace_bytes(B, K, V, N))


def best_first_tree_build(q, root_token, N, parent=None, tokens=None, depth=None, rho=None,
                          ahat=None, workspace=None, stream=None):
    """q float32 [B][K][V] marginals.  Returns (parent, tokens, depth int32
    [B][N], rho float32 [B][N], ahat float64 [B])."""
    B, K, V = q.shape
    parent = parent if parent is not None else _empty((B, N), torch.int32, q)
    tokens = tokens if tokens is not None else _empty((B, N), torch.int32, q)
    depth = depth if depth is not None else _empty((B, N), torch.int32, q)
    rho = rho if rho is not None else _empty((B, N), torch.float32, q)
    ahat = ahat if ahat is not None else _empty((B,), torch.float64, q)
    need = best_first_workspace_bytes(B, K, V, N)
    if workspace is None:
        workspace = _empty((max(need, 1),), torch.uint8, q)
    rc = lib.tsd_best_first_tree_build(
        _ptr(q, torch.float32, "q"), _ptr(root_token, torch.int32, "root_token"), B, K, V, N,
        _ptr(parent, torch.int32, "parent"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(depth, torch.int32, "depth"), _ptr(rho, torch.float32, "rho"),
        _ptr(ahat, torch.float64, "ahat"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "best_first_tree_build")
    return parent, tokens, depth, rho, ahat


# ---------------------------------------------------------------------------
# dynamic draft trees
# ---------------------------------------------------------------------------


def dynamic_tree_pool_base(level: int, k: int) -> int:
    """First pool id of an expansion level (level >= 1)."""
    return 1 if level == 1 else 1 + k + (level - 2) * k * k


def dynamic_tree_pool_size(levels: int, k: int) -> int:
    """Pool ids used by `levels` levels, root included."""
    if levels == 0:
        return 1
    return dynamic_tree_pool_base(levels, k) + (k if levels == 1 else k * k)


def dynamic_tree_new_pool(B: int, M_max: int, device):
    """Pool arrays (parent, token, depth int32, score float32), [B][M_max]."""
    i32 = dict(dtype=torch.int32, device=device)
    return (torch.empty((B, M_max), **i32), torch.empty((B, M_max), **i32),
            torch.empty((B, M_max), **i32), torch.empty((B, M_max), dtype=torch.float32,
                                                         device=device))


def dynamic_tree_workspace_bytes(B: int, F: int, k: int) -> int:
    return int(lib.tsd_dynamic_tree_workspace_bytes(B, F, k))


def dynamic_tree_expand(q, k, level, pool, root_token=None, frontier=None, next_frontier=None,
                        workspace=None, stream=None):
    """One expansion level.  q float32 [B][F][V]: the draft rows of the F
    frontier nodes (F = 1 at level 1: the root).  pool: the four [B][M_max]
    arrays (updated).  Returns the next frontier, int32 [B][k]."""
    B, F, V = q.shape
    par, tok, dep, sco = pool
    M_max = par.shape[1]
    next_frontier = next_frontier if next_frontier is not None else _empty((B, k), torch.int32, q)
    need = dynamic_tree_workspace_bytes(B, F, k)
    if workspace is None:
        workspace = _empty((max(need, 1),), torch.uint8, q)
    rc = lib.tsd_dynamic_tree_expand(
        _ptr(q, torch.float32, "q"),
        _ptr(root_token, torch.int32, "root_token") if root_token is not None else None,
        B, F, V, k, level,
        _ptr(frontier, torch.int32, "frontier") if frontier is not None else None,
        _ptr(par, torch.int32, "pool_parent"), _ptr(tok, torch.int32, "pool_token"),
        _ptr(dep, torch.int32, "pool_depth"), _ptr(sco, torch.float32, "pool_score"), M_max,
        _ptr(next_frontier, torch.int32, "next_frontier"), _ptr(workspace, None, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    _check(rc, "dynamic_tree_expand")
    return next_frontier


def dynamic_tree_rerank(pool, M, N, parent=None, tokens=None, depth=None, score=None,
                        stream=None):
    """The N-node draft tree from pool ids 0..M-1.  Returns (parent, tokens,
    depth int32 [B][N], score float32 [B][N])."""
    par, tok, dep, sco = pool
    B, M_max = par.shape
    parent = parent if parent is not None else _empty((B, N), torch.int32, par)
    tokens = tokens if tokens is not None else _empty((B, N), torch.int32, par)
    depth = depth if depth is not None else _empty((B, N), torch.int32, par)
    score = score if score is not None else _empty((B, N), torch.float32, par)
    rc = lib.tsd_dynamic_tree_rerank(
        _ptr(par, torch.int32, "pool_parent"), _ptr(tok, torch.int32, "pool_token"),
        _ptr(dep, torch.int32, "pool_depth"), _ptr(sco, torch.float32, "pool_score"), B, M, M_max,
        N, _ptr(parent, torch.int32, "parent"), _ptr(tokens, torch.int32, "tokens"),
        _ptr(depth, torch.int32, "depth"), _ptr(score, torch.float32, "score"), _stream(stream))
    _check(rc, "dynamic_tree_rerank")
    return parent, tokens, depth, score


# ---------------------------------------------------------------------------
# tree budget
# ---------------------------------------------------------------------------

def verify_step_cost(B, Hq, Hkv, D, prefix_len, V, D_max, N, hbm_gbs, tc_tflops):
    """Host-only: (bytes, flops, roofline microseconds) of one verify step with
    N-node trees.  prefix_len: a sequence of B host integers."""
    if len(prefix_len) != B:
        raise TsdError("prefix_len must hold B lengths")
    pl = (ctypes.c_int32 * B)(*[int(x) for x in prefix_len])
    out = [ctypes.c_double(), ctypes.c_double(), ctypes.c_double()]
    _check(lib.tsd_verify_step_cost(B, Hq, Hkv, D, ctypes.cast(pl, ctypes.c_void_p), V, D_max, N,
                                    float(hbm_gbs), float(tc_tflops),
                                    *[ctypes.cast(ctypes.byref(o), ctypes.c_void_p) for o in out]),
           "verify_step_cost")
    return tuple(o.value for o in out)


def budget_calibrate(t_roof, t_meas):
    """Host-only: least-squares (alpha, beta) of t_meas ~ alpha * t_roof + beta."""
    n = len(t_roof)
    x = (ctypes.c_double * n)(*[float(v) for v in t_roof])
    y = (ctypes.c_double * n)(*[float(v) for v in t_meas])
    a, b = ctypes.c_double(), ctypes.c_double()
    _check(lib.tsd_budget_calibrate(ctypes.cast(x, ctypes.c_void_p), ctypes.cast(y, ctypes.c_void_p),
                                    n, ctypes.cast(ctypes.byref(a), ctypes.c_void_p),
                                    ctypes.cast(ctypes.byref(b), ctypes.c_void_p)),
           "budget_calibrate")
    return a.value, b.value


def budget_select(rho, cost, l_ar, n_opt=None, s_opt=None, stream=None):
    """rho float32 [B][N_max] (device), cost float32 [N_max + 1] (device).
    Returns (n_opt int32 [B], s_opt float32 [B])."""
    B, N_max = rho.shape
    n_opt = n_opt if n_opt is not None else _empty((B,), torch.int32, rho)
    s_opt = s_opt if s_opt is not None else _empty((B,), torch.float32, rho)
    if cost.numel() != N_max + 1:
        raise TsdError("cost must hold N_max + 1 entries")
    _check(lib.tsd_budget_select(_ptr(rho, torch.float32, "rho"), B, N_max,
                                 _ptr(cost, torch.float32, "cost"), float(l_ar),
                                 _ptr(n_opt, torch.int32, "n_opt"),
                                 _ptr(s_opt, torch.float32, "s_opt"), _stream(stream)),
           "budget_select")
    return n_opt, s_opt


def set_option(key: int, value: int) -> None:
    """Process-wide library option (OPT_WAIT_LIMIT_NS, OPT_TEST_STALL)."""
    _check(lib.tsd_set_option(key, value), "set_option")


def get_option(key: int) -> int:
    return int(lib.tsd_get_option(key))


def version() -> str:
    return lib.tsd_version().decode()
