"""bench.py's command line on a machine without a GPU: the reference arm
(the CPU oracle) prints one JSON line with the contract's keys, other ranks
of a multi-rank launch print nothing, and the product package never reaches
the oracle."""
import json
import os
import re
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "exact_attention_forward_07_gb300")


def _run(extra_env=None, *args):
    env = dict(os.environ)
    env.update(extra_env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=env, timeout=600, cwd=ROOT)


def test_reference_arm_json_line():
    r = _run({"RANK": "0", "WORLD_SIZE": "1", "LOCAL_RANK": "0"}, "--impl", "reference",
             "--workload", "tiny_b1h1n128d64", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["steps"] == 2
    assert d["config"]["workload"] == "tiny_b1h1n128d64"
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    r = _run({"RANK": "1", "WORLD_SIZE": "2", "LOCAL_RANK": "1"}, "--impl", "reference",
             "--gpus", "2", "--workload", "tiny_b1h1n128d64", "--steps", "2", "--warmup", "3")
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_warmup_below_three_is_refused():
    r = _run(None, "--impl", "reference", "--workload", "tiny_b1h1n128d64", "--warmup", "2")
    assert r.returncode != 0


def test_product_package_does_not_use_the_oracle():
    """Only tests, the smoke check and bench.py's CPU baseline may reach the
    oracle: no source of the package or its CUDA library mentions it."""
    for dirpath, _, files in os.walk(PKG):
        for name in files:
            if not name.endswith((".py", ".cu", ".cuh", ".h")):
                continue
            text = open(os.path.join(dirpath, name), encoding="utf-8").read()
            assert not re.search(r"\boracle\b", text), os.path.join(dirpath, name)


def test_kernel_hash_ignores_comments():
    """bench.py ties a committed ncu summary to the library's code by a hash
    that skips comments and blank lines, so editing a comment keeps the
    summary's DRAM traffic in the roofline while any code change drops it."""
    sys.path.insert(0, ROOT)
    import bench
    src = "int a; // note\n/* block\n comment */\n\nint b;  \n"
    assert bench._code_only(src) == "int a;\nint b;"
    assert bench._code_only(src) == bench._code_only(src.replace("note", "other note"))
    assert bench._code_only(src) != bench._code_only(src.replace("int b", "int c"))
    assert re.fullmatch(r"[0-9a-f]{16}", bench.kernel_source_hash())
