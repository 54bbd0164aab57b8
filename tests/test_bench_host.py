"""Host-side bookkeeping of bench.py: the digest that ties a committed ncu
traffic figure to the kernel source it was taken on. No GPU."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    sys.path.insert(0, ROOT)
    import bench
    return bench


def test_digest_ignores_comments_and_layout(tmp_path, monkeypatch):
    bench = _bench()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    code = "int f(int x)\n{\n    return x + 1;  // add one\n}\n"
    (tmp_path / "a.cu").write_text(code)
    d0 = bench.source_digest("a.cu")
    (tmp_path / "a.cu").write_text("// header\n/* block\n   comment */\nint f(int x) {\n"
                                   "  return x + 1;\n}\n")
    assert bench.source_digest("a.cu") == d0          # comments and spacing only
    (tmp_path / "a.cu").write_text(code.replace("x + 1", "x + 2"))
    assert bench.source_digest("a.cu") != d0          # a code change


def test_committed_traffic_is_tied_to_its_workload_and_source(tmp_path, monkeypatch):
    bench = _bench()
    import json
    t = bench.committed_traffic("decode_kernel", "decode_b32_gqa7_ps16")
    assert t is None or t > 0                       # None once the kernel has changed
    assert bench.committed_traffic("decode_kernel", "another_workload") is None
    # a record whose digest no longer matches its source gives None
    (tmp_path / "profiles").mkdir()
    (tmp_path / "k.cu").write_text("int g() { return 1; }\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    rec = {"workload": "w", "source": "k.cu", "source_sha": bench.source_digest("k.cu"),
           "dram_bytes_per_launch": 123}
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"k": rec}))
    assert bench.committed_traffic("k", "w") == 123
    (tmp_path / "k.cu").write_text("int g() { return 2; }\n")
    assert bench.committed_traffic("k", "w") is None
