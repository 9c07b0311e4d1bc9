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


def test_clock_samples_kept_only_inside_the_timed_region(tmp_path):
    """The clock record of a bench line uses only the nvidia-smi samples whose
    timestamps fall inside the timed region, and says so when none did."""
    sys.path.insert(0, ROOT)
    import datetime
    import bench

    class _Done:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    def sampler_with(lines):
        s = bench.ClockSampler(0)
        s.out_path = str(tmp_path / "clocks.csv")
        with open(s.out_path, "w") as f:
            f.write("".join(lines))
        s.fh = open(s.out_path, "a")
        s.proc = _Done()
        return s

    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    def row(dt_s, mhz, watts, power_cap):
        ts = (t0 + datetime.timedelta(seconds=dt_s)).strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
        cap = "Active" if power_cap else "Not Active"
        return f"{ts}, 0, {mhz}, 2070, {watts}, 0x4, Not Active, Not Active, Not Active, {cap}\n"

    lines = [row(0.0, 2070, 120, False), row(1.0, 1800, 1390, True), row(1.2, 1820, 1388, True),
             row(1.4, 1790, 1391, True), row(3.0, 2070, 150, False)]
    window = ((t0 + datetime.timedelta(seconds=0.9)).timestamp(),
              (t0 + datetime.timedelta(seconds=1.5)).timestamp())
    rec = sampler_with(lines).stop(window=window)
    assert rec["samples"] == 3 and rec["sampled"] == "timed region"
    assert rec["sm_mhz"] == 1800 and rec["power_w_max"] == 1391
    assert rec["reasons"] == ["sw_power_cap"]
    # a window that no sample falls in: the whole run, marked as such
    far = (window[0] + 100, window[1] + 100)
    rec = sampler_with(lines).stop(window=far)
    assert rec["samples"] == 5 and rec["sampled"].startswith("whole run")
