"""CPU-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every function include/tsd.h declares, and the binding's signature table
matches the header.  No compute call is made (no GPU here)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "tsd.h")


@pytest.fixture(scope="module")
def lib_path():
    import __graft_entry__
    return __graft_entry__._build_module().build()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(tsd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ["tsd_tree_build_ancestors", "tsd_tree_attn_fwd", "tsd_tree_verify_greedy",
              "tsd_kv_commit_path", "tsd_best_first_tree_build"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib_path):
    lib = ctypes.CDLL(lib_path)
    for n in _declared():
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", lib_path], capture_output=True, text=True)
    exported = set(re.findall(r"\bT (tsd_[a-z_0-9]+)", out.stdout))
    assert set(_declared()) <= exported
    # nothing else of ours leaks out of the shared object
    assert exported == set(_declared())


def test_binding_signatures_match_header(lib_path):
    import tree_speculative_decoding_virtual_gb300 as tsd
    assert set(tsd.SIGNATURES) == set(_declared())
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    for name, (_, args) in tsd.SIGNATURES.items():
        m = re.search(r"\b%s\s*\((.*?)\)\s*;" % name, text, flags=re.S)
        assert m, name
        params = [p for p in m.group(1).split(",") if p.strip() and p.strip() != "void"]
        assert len(params) == len(args), (name, len(params), len(args))


def test_version_string(lib_path):
    lib = ctypes.CDLL(lib_path)
    lib.tsd_version.restype = ctypes.c_char_p
    assert lib.tsd_version().decode().startswith("tsd")


def test_host_argument_checks_without_gpu(lib_path):
    """Argument validation happens on the host before any CUDA call."""
    import tree_speculative_decoding_virtual_gb300 as tsd
    L = tsd.lib
    # N_max above the limit
    assert L.tsd_tree_build_ancestors(None, None, 1, 300, 4, None, None, None, None, None) == -2
    # null outputs
    assert L.tsd_tree_build_ancestors(None, None, 1, 8, 4, None, None, None, None, None) == -1
    # B == 0 is an empty batch: nothing to do
    assert L.tsd_tree_build_ancestors(None, None, 0, 8, 4, None, None, None, None, None) == 0
    # head dim not supported
    assert L.tsd_tree_attn_workspace_bytes(1, 8, 4, 4, 96, 100) == 0
    # key ranges longer than 32 splits of 64 key tiles of 128 keys
    assert L.tsd_tree_attn_workspace_bytes(1, 8, 4, 4, 128, 262144) > 0
    assert L.tsd_tree_attn_workspace_bytes(1, 8, 4, 4, 128, 262145) == 0
    # head dim not supported by the commit kernel
    assert L.tsd_kv_commit_path(None, None, 1, 0, None, 1, 1, None, None, None, None, None,
                                1, 8, 4, 80, 4, None, None, None, None) == -2
    # best-first budget larger than the number of distinct paths (K=1, V=3 -> 3 nodes)
    assert L.tsd_best_first_tree_build(None, None, 1, 1, 3, 5, None, None, None, None, None,
                                       None, 0, None) == -2
