"""Host logic of bench.py (CPU only): the kernel-source digest that ties
committed ncu figures to the build, and the traffic lookup that uses it."""

import os
import shutil

import pytest

import bench


def test_code_only_strips_comments_and_layout():
    src = 'int a = 1; // note\n/* block\n comment */ int  b =\n 2;\n'
    assert bench._code_only(src) == "int a = 1; int b = 2;"


def test_code_only_keeps_string_and_char_literals():
    src = 'asm("add.rn.f32 %0, %1; // not a comment\\n" : "=f"(x)); char c = \'/\'; // gone\n'
    out = bench._code_only(src)
    assert '"add.rn.f32 %0, %1; // not a comment\\n"' in out
    assert "'/'" in out
    assert "gone" not in out


def test_code_only_separates_tokens_around_block_comments():
    assert bench._code_only("int/*x*/y;") == "int y;"


@pytest.fixture
def tree(tmp_path, monkeypatch):
    """A private copy of the CUDA sources and profiles folder as bench's root."""
    root = tmp_path / "root"
    shutil.copytree(os.path.join(bench.ROOT, "tree_speculative_decoding_virtual_gb300", "csrc"),
                    root / "tree_speculative_decoding_virtual_gb300" / "csrc")
    (root / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(root))
    return root


def _edit(root, name, fn):
    p = root / "tree_speculative_decoding_virtual_gb300" / "csrc" / name
    p.write_text(fn(p.read_text()))


def test_digest_ignores_comments_but_not_code(tree):
    d0 = bench.kernel_sources_digest()
    _edit(tree, "commit.cu", lambda s: "// a new comment line\n" + s.replace("\n", "\n\n", 3))
    assert bench.kernel_sources_digest() == d0
    _edit(tree, "commit.cu", lambda s: s + "\nstatic int extra_symbol = 1;\n")
    assert bench.kernel_sources_digest() != d0


def test_traffic_lookup_follows_the_digest(tree):
    prof = tree / "profiles" / "traffic_tree_attn_fwd_8b.md"
    prof.write_text("traffic_bytes_per_launch: 123456\nkernel_sources_sha256_16: %s\n"
                    % bench.kernel_sources_digest("tree_attn_fwd"))
    assert bench.ncu_traffic("tree_attn_fwd", "8b") == 123456.0
    # another kernel's source does not detach the attention figures
    _edit(tree, "best_first.cu", lambda s: s + "\nstatic int other_kernel = 3;\n")
    assert bench.ncu_traffic("tree_attn_fwd", "8b") == 123456.0
    _edit(tree, "attention.cu", lambda s: s + "\nstatic int changed_code = 2;\n")
    assert bench.ncu_traffic("tree_attn_fwd", "8b") is None
    assert bench.ncu_traffic("tree_attn_fwd", "70b") is None  # no file


def test_kernel_sources_exist():
    csrc = os.path.join(bench.ROOT, "tree_speculative_decoding_virtual_gb300", "csrc")
    for key, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.isfile(os.path.join(csrc, n)), (key, n)



def test_reference_arm_line_contract(capsys):
    """The reference arm (the oracle timed on the host cores) prints one JSON
    line with the metric, the oracle's baseline block and a zero-copy e2e."""
    import json
    rc = bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "3", "--warmup", "3"])
    assert rc in (None, 0)
    line = [l for l in capsys.readouterr().out.strip().splitlines() if l.startswith("{")][-1]
    d = json.loads(line)
    assert d["impl"] == "reference" and d["steps"] == 3 and d["warmup"] == 3
    assert d["unit"] == "steps/s" and d["higher_is_better"] is True and d["value"] > 0
    assert d["config"]["workload"]
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
