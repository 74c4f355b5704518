"""Host-side helpers of bench.py (no GPU): the kernel-source hash that guards
the recorded ncu traffic ignores comments and blank lines but not code, and
the consumer naming follows the library's default rule."""
import json

import bench
import workloads as W


def test_code_only_drops_comments_and_blank_lines():
    src = "int a; // note\n\n/* block\n comment */ int b;  \n   \nint c;\n"
    assert bench._code_only(src) == "int a;\n int b;\nint c;"


def test_source_hash_ignores_comments_not_code(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_attention_photon_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.ATTENTION_SOURCES:
        (csrc / f).write_text("int x = 1;\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    (csrc / bench.ATTENTION_SOURCES[0]).write_text("// a comment\nint x = 1;  // same code\n")
    assert bench.kernel_source_hash() == h0
    (csrc / bench.ATTENTION_SOURCES[0]).write_text("int x = 2;\n")
    assert bench.kernel_source_hash() != h0


def test_traffic_record_is_dropped_when_the_sources_differ(tmp_path, monkeypatch):
    csrc = tmp_path / "paged_kv_attention_photon_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in bench.ATTENTION_SOURCES:
        (csrc / f).write_text("int y;\n")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"qwen_b64": {"dram_bytes_per_launch": 123, "kernel_source_sha": "0" * 16}}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("qwen_b64") is None
    rec["qwen_b64"]["kernel_source_sha"] = bench.kernel_source_hash()
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("qwen_b64") == 123


def test_consumer_names():
    assert bench.consumer_name(0, W.qwen_b64(batch=2, num_blocks=600)).startswith("tensor")
    assert bench.consumer_name(1, W.tiny()) == "CUDA cores"
    assert bench.consumer_name(2, W.tiny()) == "CUDA cores"        # tiny is fp32
