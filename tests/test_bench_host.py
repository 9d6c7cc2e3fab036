"""Host logic of bench.py that needs no GPU: the key of the committed DRAM
traffic record (the kernel code's hash) and the record lookup."""

import json
import os
import shutil

import bench


def _tree(tmp_path, files):
    d = tmp_path / "sparse_convolution_hash_gb300" / "csrc"
    d.mkdir(parents=True)
    for name, text in files.items():
        (d / name).write_text(text)
    return str(tmp_path)


def _hash(monkeypatch, root):
    monkeypatch.setattr(bench, "ROOT", root)
    return bench.kernel_source_hash()


def test_traffic_key_ignores_comments_and_layout(tmp_path, monkeypatch):
    base = "int f(int a) {\n  return a + 1;  // one more\n}\n/* block */\n"
    same = "// header comment\nint f(int a)\n{\n    return a + 1;\n}\n"
    h0 = _hash(monkeypatch, _tree(tmp_path / "a", {"k.cu": base}))
    h1 = _hash(monkeypatch, _tree(tmp_path / "b", {"k.cu": same}))
    assert h0 == h1


def test_traffic_key_changes_with_code_and_file_names(tmp_path, monkeypatch):
    base = "int f(int a) { return a + 1; }\n"
    h0 = _hash(monkeypatch, _tree(tmp_path / "a", {"k.cu": base}))
    h1 = _hash(monkeypatch, _tree(tmp_path / "b", {"k.cu": base.replace("+ 1", "+ 2")}))
    h2 = _hash(monkeypatch, _tree(tmp_path / "c", {"j.cu": base}))
    assert len({h0, h1, h2}) == 3


def test_stale_record_reads_as_missing(tmp_path, monkeypatch):
    root = tmp_path / "r"
    shutil.copytree(os.path.join(bench.ROOT, "profiles"), root / "profiles")
    _tree(root, {"k.cu": "int g() { return 0; }\n"})
    monkeypatch.setattr(bench, "ROOT", str(root))
    assert bench.measured_traffic("lidar_subm_f16", "build") is None
