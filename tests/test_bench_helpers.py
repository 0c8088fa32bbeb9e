"""bench.py's host helpers (no GPU): the code hash that decides whether a
committed ncu capture still describes a kernel, and the traffic lookup."""
import json
import os

import bench


def test_code_sha_ignores_comments_and_layout(tmp_path):
    a = tmp_path / "a.cu"
    a.write_text("__global__ void k(int* p) {\n  p[0] = 1;  // one\n}\n/* block */\n")
    b = tmp_path / "b.cu"
    b.write_text("// header\n__global__ void k(int* p) { p[0] = 1; }\n")
    c = tmp_path / "c.cu"
    c.write_text("__global__ void k(int* p) { p[0] = 2; }\n")
    assert bench.code_sha(str(a)) == bench.code_sha(str(b))
    assert bench.code_sha(str(a)) != bench.code_sha(str(c))


def test_traffic_is_null_once_the_kernel_code_changes(tmp_path, monkeypatch):
    csrc = tmp_path / "dfa_parsing_delimiter_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = csrc / "k.cu"
    src.write_text("__global__ void k() {}\n")
    entry = {"kernel": "k", "dram_bytes_per_launch": 123.0, "kernel_source": "k.cu",
             "kernel_code_sha256_prefix": bench.code_sha(str(src))}
    (tmp_path / "profiles" / "ncu_traffic.json").write_text(json.dumps({"w": entry}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench._traffic("w") == 123.0
    assert bench._traffic("other") is None
    src.write_text("// a comment only\n__global__ void k() {}\n")
    assert bench._traffic("w") == 123.0
    src.write_text("__global__ void k() { int x = 0; }\n")
    assert bench._traffic("w") is None


def test_committed_traffic_entries_name_existing_sources():
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    with open(os.path.join(root, "profiles", "ncu_traffic.json")) as f:
        d = json.load(f)
    for e in d.values():
        assert os.path.exists(os.path.join(root, "dfa_parsing_delimiter_gb300", "csrc",
                                           e["kernel_source"]))
        assert os.path.exists(os.path.join(root, e["source"]))
        assert e["dram_bytes_per_launch"] > 0
