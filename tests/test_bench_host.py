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


def _ncu_csv(path, launches):
    """An ncu --csv metrics log: one row per (launch, metric)."""
    lines = ['"ID","Kernel Name","Metric Name","Metric Unit","Metric Value"']
    for i, (name, rd, wr) in enumerate(launches):
        lines.append(f'"{i}","void spc::(anonymous namespace)::{name}(args)","dram__bytes_read.sum","Mbyte","{rd}"')
        lines.append(f'"{i}","void spc::(anonymous namespace)::{name}(args)","dram__bytes_write.sum","Kbyte","{wr}"')
        lines.append(f'"{i}","void spc::(anonymous namespace)::{name}(args)","gpu__time_duration.sum","usecond","1.0"')
    path.write_text("==PROF== header line\n" + "\n".join(lines) + "\n")


def test_traffic_record_groups_launches_by_phase(tmp_path, monkeypatch):
    """Two steps of a training workload: the build counts its table init,
    insert and probe; the conv launches alternate forward / dinput; dfilter
    counts its partial and reduction kernels; per-call bytes are the sums over
    a phase's kernels divided by its calls."""
    root = tmp_path / "r"
    (root / "profiles").mkdir(parents=True)
    _tree(root, {"k.cu": "int h() { return 1; }\n"})
    monkeypatch.setattr(bench, "ROOT", str(root))
    step = [("k_build_init", 8.0, 0.0), ("k_hash_insert", 10.0, 2000.0), ("k_map_probe_x3", 50.0, 4000.0),
            ("k_conv_tc<bf16>", 120.0, 25000.0), ("k_conv_tc<bf16>", 130.0, 30000.0),
            ("k_wgrad_tc<bf16>", 200.0, 33000.0), ("k_wgrad_reduce", 33.0, 400.0)]
    csv = tmp_path / "log.csv"
    _ncu_csv(csv, step + step)
    bench.record_traffic(str(csv), "shell192x4_train_bf16", ["build", "fwd", "dgrad", "wgrad"])
    rec = json.loads((root / "profiles" / "dram_traffic.json").read_text())
    assert rec["src_hash"] == bench.kernel_source_hash()
    got = rec["workloads"]["shell192x4_train_bf16"]
    assert got == {"build": round((8 + 10 + 50) * 1e6 + 6000e3),
                   "fwd": round(120e6 + 25000e3), "dgrad": round(130e6 + 30000e3),
                   "wgrad": round((200 + 33) * 1e6 + 33400e3)}


def test_int8_peak_follows_the_kernel_path():
    """The int8 roofline counts fp16 products per int8 product as conv_i8
    dispatches: one on the several-accumulator path, two on the weight split."""
    assert bench.int8_fp16_products(27, 128, 128) == 1   # 54 stages, 4 accumulators of 128
    assert bench.int8_fp16_products(27, 64, 64) == 1     # 27 stages, 2 accumulators
    assert bench.int8_fp16_products(27, 256, 64) == 1    # 108 stages, 8 accumulators of 64
    assert bench.int8_fp16_products(27, 256, 128) == 1   # 108 stages: 8 accumulators of 64
    assert bench.int8_fp16_products(8, 1024, 128) == 2   # 128 stages: the split
    assert bench.int8_fp16_products(1, 8192, 64) == 2    # 128 stages: the split
    p = bench.Phase("fwd", None, "conv", 1e6, flops=1e12)
    p.fp16_per_int8 = 1
    full = bench.roofline(p, 1.0, 6000.0, 1900.0, 60.0, "i8", False)
    p.fp16_per_int8 = 2
    half = bench.roofline(p, 1.0, 6000.0, 1900.0, 60.0, "i8", False)
    assert full["peak"] == 1900.0 and half["peak"] == 950.0
    assert abs(half["frac"] - 2 * full["frac"]) < 1e-3
