"""Host-side helpers of bench.py: the source hash that decides whether the
committed DRAM-traffic figure still describes the expert-GEMM code, the lookup
of that figure, and the whole-job value over replicas."""
import json
import os
import shutil

import pytest

import bench

FILES = ("ffn_gemm.cu", "ffn_gemm_2cta.cu", "ffn_gemm_mx.cu", "device.cuh", "internal.h")


@pytest.fixture()
def tree(tmp_path, monkeypatch):
    """A copy of the hashed sources and of profiles/ under a scratch root."""
    csrc = tmp_path / "moe_expert_layer_02_gb300" / "csrc"
    csrc.mkdir(parents=True)
    src = os.path.join(bench.ROOT, "moe_expert_layer_02_gb300", "csrc")
    for n in FILES:
        shutil.copy(os.path.join(src, n), csrc / n)
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(tree, name, fn):
    p = tree / "moe_expert_layer_02_gb300" / "csrc" / name
    p.write_text(fn(p.read_text()))


def test_source_sha_ignores_comments_and_whitespace(tree):
    base = bench.source_sha()
    _edit(tree, "ffn_gemm.cu", lambda s: "// a new comment line\n" + s.replace("\n", "\n\n", 3))
    _edit(tree, "internal.h", lambda s: s + "\n/* a block\n   comment */\n")
    assert bench.source_sha() == base


def test_source_sha_follows_code(tree):
    base = bench.source_sha()
    _edit(tree, "device.cuh", lambda s: s + "\nnamespace moe { constexpr int kProbe = 1; }\n")
    assert bench.source_sha() != base


def test_kernel_traffic_only_for_the_current_source(tree):
    path = tree / "profiles" / "ffn1_decode.json"
    path.write_text(json.dumps({"source_sha": bench.source_sha(), "dram_bytes_per_launch": 123.0}))
    assert bench.kernel_traffic("ffn1", "decode") == 123.0
    assert bench.kernel_traffic("ffn1", "prefill") is None  # no summary for that workload
    _edit(tree, "ffn_gemm.cu", lambda s: s + "\nnamespace moe { constexpr int kProbe = 2; }\n")
    assert bench.kernel_traffic("ffn1", "decode") is None  # code changed since the capture


def test_replica_value_single_rank():
    value, ms = bench.replica_value(12.5, 2.0, 1)
    assert ms == 2.0 and value == pytest.approx(12.5 / 2.0e-3)


def test_source_sha_reads_only_the_argument_struct_of_internal_h(tree):
    # declarations of other kernels do not change the expert GEMM; a field of
    # the struct it reads does
    base = bench.source_sha()
    _edit(tree, "internal.h", lambda s: s + "\nnamespace moe { int some_other_launcher(int); }\n")
    assert bench.source_sha() == base
    _edit(tree, "internal.h", lambda s: s.replace("struct GroupedFfnArgs {",
                                                  "struct GroupedFfnArgs {\n  int probe_field;", 1))
    assert bench.source_sha() != base


def test_kernel_traffic_follows_the_files_a_summary_names(tree):
    # a summary of the SM-pair GEMM names its own source; editing another
    # kernel's file leaves it valid, editing its own does not
    pair = ("ffn_gemm_2cta.cu", "device.cuh", "internal.h")
    (tree / "profiles" / "ffn1_prefill.json").write_text(json.dumps(
        {"source_files": list(pair), "source_sha": bench.source_sha(pair),
         "dram_bytes_per_launch": 7.0}))
    (tree / "profiles" / "ffn1_decode.json").write_text(json.dumps(
        {"source_sha": bench.source_sha(), "dram_bytes_per_launch": 5.0}))
    _edit(tree, "ffn_gemm.cu", lambda s: s + "\nnamespace moe { constexpr int kProbe = 3; }\n")
    assert bench.kernel_traffic("ffn1", "prefill") == 7.0
    assert bench.kernel_traffic("ffn1", "decode") is None
    _edit(tree, "ffn_gemm_2cta.cu", lambda s: s + "\nnamespace moe { constexpr int kProbe = 4; }\n")
    assert bench.kernel_traffic("ffn1", "prefill") is None

