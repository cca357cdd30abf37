"""Structure checks that need no GPU: the product path never reaches the oracle,
and the bench helpers that pick workloads and attach ncu traffic behave."""
import argparse
import ast
import hashlib
import json
import os

import bench
import tq_synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "vector_quantization_02_b300")


def _imports(path):
    tree = ast.parse(open(path).read())
    for node in ast.walk(tree):
        if isinstance(node, ast.Import):
            for a in node.names:
                yield node, a.name
        elif isinstance(node, ast.ImportFrom):
            yield node, node.module or ""


def test_product_package_never_imports_the_oracle():
    for dirpath, _, files in os.walk(PKG):
        for f in files:
            if f.endswith(".py"):
                for _, name in _imports(os.path.join(dirpath, f)):
                    assert not name.split(".")[0] == "oracle", f"{f} imports {name}"
    # and the native sources do not include anything from it
    for f in os.listdir(os.path.join(PKG, "csrc")):
        text = open(os.path.join(PKG, "csrc", f), errors="ignore").read()
        assert "oracle/" not in text and "tq_oracle" not in text, f


def test_bench_reaches_the_oracle_only_in_its_cpu_legs():
    path = os.path.join(ROOT, "bench.py")
    tree = ast.parse(open(path).read())
    allowed = {"oracle_throughput"}
    for fn in ast.walk(tree):
        if isinstance(fn, ast.FunctionDef):
            for node in ast.walk(fn):
                if isinstance(node, ast.ImportFrom) and (node.module or "").startswith("oracle"):
                    assert fn.name in allowed, f"oracle imported in {fn.name}"
    # no module-level import of it either
    for node in tree.body:
        if isinstance(node, (ast.Import, ast.ImportFrom)):
            names = [a.name for a in node.names] if isinstance(node, ast.Import) else [node.module or ""]
            assert not any(n.startswith("oracle") for n in names)


def test_reduced_workload_keeps_the_shape_and_caps_tokens():
    base = tq_synth.WORKLOADS["vector_search_1m"]
    w = bench.workload(argparse.Namespace(workload="vector_search_1m", tokens=100000))
    assert w.N == 100000 and (w.G, w.H, w.d, w.name) == (base.G, base.H, base.d, base.name)
    assert bench.workload(argparse.Namespace(workload="vector_search_1m", tokens=0)).N == base.N
    assert bench.workload(argparse.Namespace(workload="single_head_3bit", tokens=10 ** 9)).N == \
        tq_synth.WORKLOADS["single_head_3bit"].N


def test_traffic_is_reported_only_for_the_captured_source_and_workload(tmp_path, monkeypatch):
    src = "k_score_tc.cu"
    sha = hashlib.sha256(open(os.path.join(PKG, "csrc", src), "rb").read()).hexdigest()[:16]
    f = tmp_path / "traffic.json"
    f.write_text(json.dumps({"score_tc": {"dram_bytes_per_launch": 123, "source_sha": sha,
                                          "workload": "qwen25_3b_decode"}}))
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.kernel_traffic("score_tc", src, "qwen25_3b_decode") == 123
    assert bench.kernel_traffic("score_tc", src, "long_context_131k") is None
    assert bench.kernel_traffic("encode_tc", "k_encode_tc.cu", "qwen25_3b_decode") is None
    f.write_text(json.dumps({"score_tc": {"dram_bytes_per_launch": 123, "source_sha": "0" * 16,
                                          "workload": "qwen25_3b_decode"}}))
    assert bench.kernel_traffic("score_tc", src, "qwen25_3b_decode") is None
    # an entry kernel@workload serves that workload; the kernel's own entry the one it names
    f.write_text(json.dumps({
        "score_tc": {"dram_bytes_per_launch": 123, "source_sha": sha, "workload": "qwen25_3b_decode"},
        "score_tc@llama31_8b_prefill": {"dram_bytes_per_launch": 456, "source_sha": sha,
                                        "workload": "llama31_8b_prefill"}}))
    assert bench.kernel_traffic("score_tc", src, "qwen25_3b_decode") == 123
    assert bench.kernel_traffic("score_tc", src, "llama31_8b_prefill") == 456
    assert bench.kernel_traffic("score_tc", src, "long_context_131k") is None


def test_committed_traffic_entries_name_existing_summaries():
    t = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    for k, v in t.items():
        if k.startswith("_"):
            continue
        assert os.path.exists(os.path.join(ROOT, v["summary"])), v["summary"]
        assert v["dram_bytes_per_launch"] > 0 and v["workload"] in tq_synth.WORKLOADS


def test_both_bench_arms_report_the_same_workload_config():
    w = tq_synth.WORKLOADS["vector_search_1m"]
    c = bench.workload_config(w, "mse", 4, "hadamard")
    assert c == {"workload": w.name, "mode": "mse", "G": w.G, "N": w.N, "H": w.H, "d": w.d, "bits": 4,
                 "key_dtype": "float32", "top_k": w.top_k, "rotation": "hadamard"}
    # both arms print exactly this dict as their config (how L2 was handled is a separate key)
    src = open(os.path.join(ROOT, "bench.py")).read()
    assert src.count('"config": workload_config(w, args.mode, bits, args.rotation)') == 2
