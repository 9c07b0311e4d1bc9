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
    assert bench.kernel_source_hash("fa_bwd_kernel") != bench.kernel_source_hash("fa_fwd_kernel")


def test_clock_samples_kept_only_inside_the_timed_region():
    """The clock record of a bench line uses only the samples whose host
    timestamps fall inside the timed region, and says so when none did;
    reason bits decode to NVML's clock-event names."""
    sys.path.insert(0, ROOT)
    import bench

    s = bench.ClockSampler(reader=lambda: None)
    s.samples = [(0.0, 2070.0, 2070.0, 120.0, 0x0), (1.0, 1800.0, 2070.0, 1390.0, 0x4),
                 (1.2, 1820.0, 2070.0, 1388.0, 0x4), (1.4, 1790.0, 2070.0, 1391.0, 0x4 | 0x1),
                 (3.0, 2070.0, 2070.0, 150.0, 0x0)]
    rec = s.stop(window=(0.9, 1.5))
    assert rec["samples"] == 3 and rec["sampled"] == "timed region"
    assert rec["sm_mhz"] == 1800 and rec["power_w_max"] == 1391
    assert rec["reasons"] == ["sw_power_cap"]
    # a window that no sample falls in: the whole run, marked as such
    rec = s.stop(window=(100.0, 101.0))
    assert rec["samples"] == 5 and rec["sampled"].startswith("whole run")
    s.samples = [(1.0, 1500.0, 2070.0, 1300.0, 0x8 | 0x20 | 0x40)]
    rec = s.stop(window=(0.0, 2.0))
    assert rec["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_thread_polls_during_a_window():
    """The background thread reads the clock source repeatedly: a 60 ms
    window at the 2 ms period holds many samples."""
    sys.path.insert(0, ROOT)
    import time as _time
    import bench

    s = bench.ClockSampler(reader=lambda: (1965.0, 2070.0, 900.0, 0x4), period_s=0.002)
    s.start()
    _time.sleep(0.02)
    t0 = _time.time()
    _time.sleep(0.06)
    t1 = _time.time()
    rec = s.stop(window=(t0, t1))
    assert rec["sampled"] == "timed region" and rec["samples"] >= 5
    assert rec["sm_mhz"] == 1965.0 and rec["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler(reader=None).stop()["reasons"] == ["NVML unavailable"]


def test_default_workload_is_the_largest_bf16_shape():
    """The line the benchmark prints by default is on the largest bf16
    target shape (the long causal sequence), and a profile summary name is
    derived from the workload it covers."""
    sys.path.insert(0, ROOT)
    import bench
    from attn_inputs import WORKLOADS
    w = WORKLOADS[bench.DEFAULT_WORKLOAD]
    bf16 = [x for x in WORKLOADS.values() if x.dtype == "bf16"]
    assert w.flops() == max(x.flops() for x in bf16 if x.name != "b16h32n8192d128_causal")
    assert (w.B, w.H, w.N, w.d, w.causal) == (1, 32, 16384, 128, True)
    assert bench.profile_summary(w.name).endswith("fa_fwd_kernel_b1h32n16384d128_causal.md")
