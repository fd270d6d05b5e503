"""bench.py's use of a committed ncu capture: the recorded DRAM bytes count only while the kernel
sources hash to the value stored beside them. The hash leaves comments out (a comment edit does
not change the kernel), and any change of code changes it."""
import json
import os

import bench
import moe_workloads as mw


def test_code_only_drops_comments_and_blank_lines():
    src = "int a = 1;  // one\n\n/* block\n   comment */ int b = 2;\n   \n// whole line\nint c = a + b;\n"
    assert bench._code_only(src) == "int a = 1;\nint b = 2;\nint c = a + b;"


def test_comment_edit_keeps_the_hash_and_code_edit_changes_it(tmp_path, monkeypatch):
    csrc = tmp_path / "routed_expert_ffn_softmax_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text("__global__ void k(int* p) {  // writes one\n  p[0] = 1;\n}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash(("k.cu",))
    (csrc / "k.cu").write_text("// a kernel\n__global__ void k(int* p) {\n  /* one */ p[0] = 1;\n}\n")
    assert bench.kernel_source_hash(("k.cu",)) == h0
    (csrc / "k.cu").write_text("__global__ void k(int* p) {\n  p[0] = 2;\n}\n")
    assert bench.kernel_source_hash(("k.cu",)) != h0


def test_recorded_traffic_only_while_the_hash_matches(tmp_path, monkeypatch):
    csrc = tmp_path / "routed_expert_ffn_softmax_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_text("int x;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash(("k.cu",))
    rec = {"w": {"kernel_source_hash": h, "dram_bytes_per_launch": 123.0}}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("w", ("k.cu",)) == 123.0
    (csrc / "k.cu").write_text("int y;\n")
    assert bench.recorded_traffic("w", ("k.cu",)) is None
    assert bench.recorded_traffic("other", ("k.cu",)) is None


def test_committed_captures_match_the_current_kernels():
    """Every committed expert, decode-step and attention capture was taken on the kernels now in the tree."""
    with open(os.path.join(bench.ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    for name, e in rec.items():
        if name.endswith("_attn"):
            sources = bench.ATTN_SOURCES
        elif e.get("sources") == "DECODE_SOURCES":  # the one-launch decode step
            sources = bench.DECODE_SOURCES
        else:
            sources = bench.expert_sources(mw.CONFIGS[name.rsplit("_T", 1)[0]].wtype)
        assert e["kernel_source_hash"] == bench.kernel_source_hash(sources), name
