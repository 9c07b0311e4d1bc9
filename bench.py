"""Throughput benchmark of the attention forward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--variant stages=S,exp_split=E]
    python bench.py --sweep [--workload NAME] [--steps K] [--sweep-reps R]
    python bench.py --rescale-stats [--workload NAME]

A step is one forward (O and LSE) over the whole workload; by default the
largest bf16 shape of the target set, the long causal sequence
[B=1, H=32, N=16384, d=128] with seeded N(0,1) inputs.  Prints one JSON
line (rank 0).  The metric is TFLOPS with 4*B*H*N^2*d FLOPs per step
(halved when causal).

Timing: W warm-up steps, then exactly K steps between a barrier and a
device synchronisation on both sides, timed with CUDA events on the stream
the kernel is launched on; the maximum over ranks is reported.  Without
--steps, K is set from the warm-up timing so the timed region lasts about
2 s (50 to 20000 steps; the largest K over ranks).  SM clock, power and
clock-event reasons are read from NVML every 2 ms on a background thread
and only the samples taken inside the timed region are kept (about ten in a
20-step run of the default workload).  The roofline's peak is the measured
burst bf16 rate for a timed region under a second and the sustained one
for longer runs (the board reaches its power limit within about a second).
Q+K+V (384 MiB for the default) exceed the 126 MB L2, so no flush is needed
between steps.  Under torchrun each rank runs the same workload on its own
GPU (heads are independent: weak scaling, no data-path collective).

`e2e` repeats the measurement through the C ABI's host-buffer entry point
(fa_fwd_host) with pinned host buffers: every step copies Q, K, V
host->device, runs the forward and copies O and LSE back, all inside the
timed region (the library overlaps the copies of one chunk of heads with
the forward of another).

`--variant` times one of the library's kernel variants (fa_fwd_variant:
K/V ring depth, share of exponentials on the FMA pipes; with --pass bwd,
fa_bwd_variant's cta_pairs) instead of the default.  `--sweep` times every variant built for the workload's head dim
and dtype, R rounds in alternating order, and prints a Markdown table of
median TFLOPS, median SM clock and FLOP per SM clock (the clock-normalised
rate, which removes the power limit's effect on the clock).
`--rescale-stats` runs the counting build once and prints how often the
online softmax's O rescale fired.  `host_us_per_call` in the line is the
host time to enqueue one call through the Python binding, measured over
the first 20 calls of the timed launch loop (a long run's later calls wait
for room in the launch queue);
`host_us_per_call_c_abi` the same for 50 direct C-ABI calls (argument
checks, cached tensor maps, launch).

`--pass bwd` times the backward pass instead (fa_bwd: dQ, dK, dV from the
forward's O and LSE and a seeded output gradient, three kernels per step;
10*B*H*N^2*d FLOPs per step, halved when causal: the five matrix products
of the gradients), with the backward oracle as its CPU baseline.

`--impl reference` times the CPU oracle (the reference arm: a plain fp64
C implementation of the definition) on the host cores, each step a bounded
sample of the same workload (128 query rows of one head).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from attn_inputs import WORKLOADS, make_workload_inputs  # noqa: E402

METRIC = "attention fwd TFLOPS (bf16, 1×GB300) and fraction of dense tensor-core peak"
METRIC_BWD = "attention bwd TFLOPS (bf16, 1×GB300) and fraction of dense tensor-core peak"
DEFAULT_WORKLOAD = "b1h32n16384d128_causal"
FALLBACK_BF16_TFLOPS = 1900.0
# The library sources each profiled kernel is built from (its launch, its
# device code and the PTX wrappers): a change to the backward's kernel file
# leaves the forward's profiles valid.
KERNEL_SOURCES = {
    "fa_fwd_kernel": ["fa_api.cu", "fa_kernel.cuh", "ptx.cuh"],
    "fa_bwd_kernel": ["fa_api.cu", "fa_kernel.cuh", "fa_bwd_kernel.cuh", "ptx.cuh"],
}
AUTO_TIMED_S = 2.0  # timed work with no --steps
SUSTAINED_AFTER_S = 1.0  # timed regions at least this long compare against the sustained peak
CPU_SAMPLE_FLOP = 1.1e12  # oracle work of the default cpu_baseline sample (~17 s on 16 cores)


def profile_summary(workload: str, kernel: str = "fa_fwd_kernel") -> str:
    """The committed ncu summary of a kernel on a workload."""
    return os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def _code_only(text: str) -> str:
    """The source without comments and blank lines (no string literal in
    these files holds a comment marker)."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_source_hash(kernel: str = "fa_fwd_kernel") -> str:
    """Hash of the code `kernel` is built from (comments excluded): a profile
    taken at one hash describes every source with the same hash."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_attention_forward_07_gb300", "csrc", name)) as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str, kernel: str = "fa_fwd_kernel"):
    """DRAM bytes per launch from the committed ncu summary of `kernel` on
    `workload`, or None when there is none or the kernel sources changed
    since that capture."""
    try:
        text = open(profile_summary(workload, kernel)).read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    m_traffic = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    if not (m_hash and m_traffic) or m_hash.group(1) != kernel_source_hash(kernel):
        return None
    return float(m_traffic.group(1))


def measured_peaks(sustained: bool = False):
    """(bf16 TFLOP/s, description): the measured burst or sustained
    cuBLAS rate, else the fallback figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    key = "bf16_tflops_sustained" if sustained else "bf16_tflops"
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), f"{key}, measured"
    except (OSError, KeyError, ValueError):
        return (1700.0 if sustained else FALLBACK_BF16_TFLOPS), f"{key}, fallback"


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class NvmlReader:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the
    driver; no Python package needed): SM clock, its maximum, board power
    and the active clock-event reasons of one GPU.  Nothing is set."""

    def __init__(self, pci_bus_id=None, index=0):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        rc = 1
        if pci_bus_id:
            rc = self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(),
                                                           ctypes.byref(self.h))
        if rc != 0:
            rc = self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
        if rc != 0:
            raise OSError("no NVML handle for the GPU")
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self.reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_mhz = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, 1)

    def _uint(self, fn, *args):
        v = self.ct.c_uint(0)
        return float(v.value) if fn(self.h, *args, self.ct.byref(v)) == 0 else None

    def __call__(self):
        """(sm_mhz, sm_max_mhz, power_w, reason bits)"""
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, 1)  # NVML_CLOCK_SM
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        bits = self.ct.c_ulonglong(0)
        ok = self.reasons_fn(self.h, self.ct.byref(bits)) == 0
        return sm, self.max_mhz, (mw / 1000.0 if mw is not None else None), (
            bits.value if ok else None)


class ClockSampler:
    """SM clock, power and clock-event reasons sampled every `period_s`
    (2 ms by default, read-only NVML) on a background thread while the
    benchmark runs; stop() keeps the samples whose host timestamps fall
    inside a given window (the timed region), so idle time around it does
    not count.  A 20-step timed region of a millisecond kernel then still
    holds about ten samples."""

    def __init__(self, reader, period_s=0.002):
        self.reader = reader
        self.period_s = period_s
        self.samples = []  # (host time, sm_mhz, sm_max_mhz, power_w, reason bits)
        self._stop = None
        self._thread = None

    @classmethod
    def for_device(cls, dev_index: int):
        import torch
        props = torch.cuda.get_device_properties(dev_index)
        bus = None
        if hasattr(props, "pci_bus_id"):
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                         getattr(props, "pci_device_id", 0))
        try:
            return cls(NvmlReader(bus, dev_index))
        except (OSError, AttributeError):
            return cls(None)

    def start(self):
        import threading
        if self.reader is None:
            return
        self._stop = threading.Event()

        def loop():
            while not self._stop.is_set():
                t = time.time()
                try:
                    self.samples.append((t, *self.reader()))
                except Exception:  # a failed read only loses that sample
                    pass
                self._stop.wait(self.period_s)

        self._thread = threading.Thread(target=loop, daemon=True)
        self._thread.start()

    def stop(self, window=None):
        """window: (start, end) host times (time.time()) to keep samples from."""
        if self.reader is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["NVML unavailable"],
                    "source": None}
        if self._thread is not None:
            self._stop.set()
            self._thread.join(timeout=5)
        rows = self.samples
        inside = [r for r in rows if window is None or window[0] <= r[0] <= window[1]]
        scope = "timed region" if inside or window is None else \
            "whole run (none inside the timed region)"
        if inside:
            rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"],
                    "source": "nvml"}
        sm = [r[1] for r in rows if r[1] is not None]
        smax = [r[2] for r in rows if r[2] is not None]
        power = [r[3] for r in rows if r[3] is not None]
        reasons = sorted({name for r in rows if r[4] is not None
                          for bit, name in _NVML_REASONS.items() if r[4] & bit})
        busy = [s for s in sm if smax and s >= 0.3 * max(smax)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(rows), "sampled": scope, "reasons": reasons,
                "source": f"nvml every {self.period_s * 1e3:g} ms"}


L2_BYTES = 126 * 1024 * 1024


def l2_note(w) -> str:
    qkv = 3 * w.B * w.H * w.N * w.d * 2
    if qkv > L2_BYTES:
        return f"no flush: Q+K+V ({qkv / 2**20:.0f} MiB) exceed the 126 MB L2"
    return (f"L2-resident: Q+K+V ({qkv / 2**20:.1f} MiB) fit in L2 and are not flushed "
            "between steps")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_step: float, steps: int, ms_local: float, world: int):
    """Whole-job TFLOPS: every rank ran `steps` steps of `flops_per_step`; the
    job took as long as its slowest rank.  Returns (tflops, ms_max)."""
    ms_max = max_over_ranks(ms_local, world)
    return world * flops_per_step * steps / (ms_max * 1e-3) / 1e12, ms_max


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def oracle_sample(w, q, k, v, n_heads: int, rows_per_head=None):
    """Time the oracle on a bounded sample: all (or `rows_per_head`) query
    rows of `n_heads` heads.  Returns (TFLOPS, seconds, description)."""
    import numpy as np
    import oracle
    BH = w.B * w.H
    heads = list(range(min(n_heads, BH)))
    sub = [x.reshape(BH, 1, w.N, w.d)[heads].reshape(1, len(heads), w.N, w.d) for x in (q, k, v)]
    if rows_per_head is None:
        rows = np.arange(len(heads) * w.N, dtype=np.int64)
    else:
        rows = np.concatenate([h * w.N + np.arange(rows_per_head[0], rows_per_head[1])
                               for h in range(len(heads))]).astype(np.int64)
    i = rows % w.N
    keys = (i + 1) if w.causal else np.full_like(i, w.N)
    flops = float(np.sum(4.0 * keys * w.d))
    sub64 = [oracle._as_f64(x) for x in sub]  # upcast outside the timed region
    t0 = time.perf_counter()
    oracle.attn_fwd(*sub64, w.causal, w.scale, rows=rows, nthreads=cpu_cores())
    dt = time.perf_counter() - t0
    desc = (f"{len(rows)} query rows ({len(heads)} head(s) x "
            f"{'all' if rows_per_head is None else rows_per_head[1] - rows_per_head[0]} rows) "
            f"of {w.name}, fp64, {cpu_cores()} threads")
    return flops / dt / 1e12, dt, desc


def bwd_output_grad(w):
    """The output gradient of the backward benchmark: N(0,1) from its own
    seeded generator, in the workload's 16-bit type."""
    import torch
    g = torch.Generator(device="cpu")
    g.manual_seed(10 * w.index + 7)
    return torch.randn((w.B, w.H, w.N, w.d), generator=g, dtype=torch.float32).to(
        w.torch_dtype)


def oracle_bwd_sample(w, q, k, v, do, n_heads: int):
    """Time the backward oracle on the first `n_heads` heads (every row).
    Returns (TFLOPS at the metric's 10*N^2*d per head, seconds, description)."""
    import oracle
    BH = w.B * w.H
    heads = min(n_heads, BH)
    sub = [oracle._as_f64(x.reshape(BH, 1, w.N, w.d)[:heads].reshape(1, heads, w.N, w.d))
           for x in (q, k, v, do)]
    t0 = time.perf_counter()
    oracle.attn_bwd(*sub, w.causal, w.scale, nthreads=cpu_cores())
    dt = time.perf_counter() - t0
    flops = 10.0 * heads * w.N * w.N * w.d / (2 if w.causal else 1)
    desc = (f"backward of {heads} head(s) x all rows of {w.name}, fp64, "
            f"{min(heads, cpu_cores())} threads (one per head)")
    return flops / dt / 1e12, dt, desc


def run_reference(args, w):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    q, k, v = make_workload_inputs(w)
    BH = w.B * w.H
    tiles = (w.N + 127) // 128
    oracle_sample_step(w, q, k, v, 0, BH, tiles)  # fp64 head copies, untimed
    for i in range(args.warmup):
        oracle_sample_step(w, q, k, v, i, BH, tiles)
    flops = 0.0
    t0 = time.perf_counter()
    for i in range(args.steps):
        flops += oracle_sample_step(w, q, k, v, args.warmup + i, BH, tiles)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(w.describe(), sample="128 query rows of one head per step"),
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": cpu_cores(),
                         "kind": "oracle",
                         "sample": f"each step: 128 consecutive query rows of one head of "
                                   f"{w.name} (fp64 C oracle, {cpu_cores()} threads)"},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


_ref_heads = {}


def oracle_sample_step(w, q, k, v, i, BH, tiles):
    """One reference step: 128 consecutive query rows of one head (cycling
    over up to 8 heads whose fp64 copies are made before timing starts)."""
    import numpy as np
    import oracle
    if not _ref_heads:
        for h in range(min(8, BH)):
            _ref_heads[h] = [oracle._as_f64(x.reshape(BH, 1, w.N, w.d)[h:h + 1].reshape(
                1, 1, w.N, w.d)) for x in (q, k, v)]
    sub = _ref_heads[i % len(_ref_heads)]
    tile = (i * 3) % tiles
    lo, hi = tile * 128, min(w.N, tile * 128 + 128)
    rows = np.arange(lo, hi, dtype=np.int64)
    keys = (rows + 1) if w.causal else np.full_like(rows, w.N)
    oracle.attn_fwd(*sub, w.causal, w.scale, rows=rows, nthreads=cpu_cores())
    return float(np.sum(4.0 * keys * w.d))


def run_ours(args, w):
    import torch

    import exact_attention_forward_07_gb300 as fa

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else torch.cuda.current_device())
    torch.cuda.set_device(dev)
    q_h, k_h, v_h = make_workload_inputs(w)
    q, k, v = (x.to(dev) for x in (q_h, k_h, v_h))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    call = fa.fa_fwd if w.dtype == "bf16" else fa.fa_fwd_fp16
    variant = parse_variant(args.variant)
    bwd = args.pass_ == "bwd"
    if variant and ("cta_pairs" in variant) != bwd:
        raise ValueError("cta_pairs is the backward's variant key (with --pass bwd), "
                         "stages/exp_split/causal_order the forward's")
    if variant and not bwd:
        def call(q, k, v, o, lse, causal, stream):  # noqa: F811
            fa.fa_fwd_variant(q, k, v, o, lse, causal=causal, stream=stream, **variant)
    stream = torch.cuda.current_stream(dev)
    flops = w.flops()
    if bwd:
        # the forward once (untimed) for O and LSE; each step is fa_bwd
        o_f, lse_f = fa.forward(q, k, v, causal=w.causal, stream=stream)
        do_h = bwd_output_grad(w)
        do = do_h.to(dev)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        ws = torch.empty(fa.fa_bwd_workspace_size(w.B, w.H, w.N, w.d), dtype=torch.uint8,
                         device=dev)

        def call(q, k, v, o, lse, causal, stream):  # noqa: F811
            fa.fa_bwd(q, k, v, o_f, lse_f, do, dq, dk, dv, ws, causal=causal, stream=stream,
                      cta_pairs=variant.get("cta_pairs"))
        flops = 2.5 * w.flops()

    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.warmup):
        if i == 1:
            w0.record(stream)
        call(q, k, v, o, lse, causal=w.causal, stream=stream)
    w1.record(stream)
    torch.cuda.synchronize(dev)
    if args.steps is None:
        # about 2 s of timed work
        t_step = w0.elapsed_time(w1) / (args.warmup - 1) * 1e-3
        steps = int(min(20000, max(50, math.ceil(AUTO_TIMED_S / max(t_step, 1e-7)))))
        args.steps = int(max_over_ranks(float(steps), world))
    status = fa.fa_get_status(stream)
    if status != 0:
        raise RuntimeError(f"kernel status {status}: {fa.fa_strerror(status)}")

    sampler = ClockSampler.for_device(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.05)
    # ---------------------------------------------------------- timed region
    barrier(world)
    torch.cuda.synchronize(dev)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    t_begin = time.time()
    ev0.record(stream)
    h0 = time.perf_counter()
    n_host = min(args.steps, 20)  # later calls of a long run wait for room in the launch queue
    for it in range(args.steps):
        call(q, k, v, o, lse, causal=w.causal, stream=stream)
        if it + 1 == n_host:
            host_us = (time.perf_counter() - h0) / n_host * 1e6  # enqueue time per call
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_end = time.time()
    barrier(world)
    # ------------------------------------------------------------------------
    clocks = sampler.stop(window=(t_begin, t_end))
    ms_local = ev0.elapsed_time(ev1)
    value, ms_total = job_throughput(flops, args.steps, ms_local, world)
    ms_step = ms_total / args.steps
    kernel_tflops = flops / (ms_local / args.steps * 1e-3) / 1e12
    status = fa.fa_get_status(stream)
    if status != 0:
        raise RuntimeError(f"kernel status {status}: {fa.fa_strerror(status)}")
    # The library's own enqueue cost: the C ABI called through ctypes with
    # its arguments built beforehand (forward, default variant), 50 calls.
    c_abi_us = None
    if not bwd and not variant:
        import ctypes
        fn = fa.lib().fa_fwd if w.dtype == "bf16" else fa.lib().fa_fwd_fp16
        cargs = (q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                 w.B, w.H, w.N, w.d, int(w.causal), ctypes.c_float(w.scale),
                 ctypes.c_void_p(stream.cuda_stream))
        torch.cuda.synchronize(dev)
        h0 = time.perf_counter()
        for _ in range(50):
            fn(*cargs)
        c_abi_us = (time.perf_counter() - h0) / 50 * 1e6
        torch.cuda.synchronize(dev)

    # ------------------------------------------------ end to end, host buffers
    # Pinned host Q, K, V in; pinned host O, LSE out; every step is one
    # fa_fwd_host call, which copies the inputs host->device, runs the forward
    # and copies the outputs back, with the copies of one chunk of heads
    # overlapping the forward of another.  Timed on the host clock around
    # fully synchronised steps.
    e2e = None
    if not args.no_e2e and not bwd:
        pin = [x.pin_memory() for x in (q_h, k_h, v_h)]
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        n_e2e = max(1, min(args.steps, args.e2e_steps))
        n_chunks = max(1, min(args.e2e_chunks, w.B * w.H))

        def e2e_step():
            fa.fa_fwd_host(*pin, o_h, lse_h, causal=w.causal, scale=w.scale, chunks=n_chunks)

        for _ in range(min(3, args.warmup) or 1):
            e2e_step()
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_local_ms = (time.perf_counter() - t0) * 1e3
        barrier(world)
        e2e_value, e2e_ms = job_throughput(flops, n_e2e, e2e_local_ms, world)
        h2d = sum(x.numel() * x.element_size() for x in pin)
        d2h = o_h.numel() * o_h.element_size() + lse_h.numel() * lse_h.element_size()
        e2e = {"value": e2e_value, "unit": "TFLOPS",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": e2e_ms / n_e2e, "chunks": n_chunks, "api": "fa_fwd_host",
               "timing": "host clock around synchronised steps"}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    # The time and the clock it ran at: milliseconds x median MHz per step
    # (thousands of SM cycles) and the FLOP each SM did per cycle.
    if clocks.get("sm_mhz"):
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        clocks["ms_per_step_x_mhz"] = ms_local / args.steps * clocks["sm_mhz"]
        clocks["flop_per_clock_per_sm"] = flops / (
            ms_local / args.steps * 1e-3 * clocks["sm_mhz"] * 1e6 * n_sm)
    sustained = ms_local * 1e-3 >= SUSTAINED_AFTER_S
    peak, peak_kind = measured_peaks(sustained)
    roofline = {"bound": "tensor", "achieved": kernel_tflops, "peak": peak,
                "unit": "TFLOP/s", "frac": kernel_tflops / peak,
                "peak_source": peak_kind + (" (timed region >= 1 s)" if sustained else
                                            " (timed region < 1 s)"),
                "traffic": profiled_traffic(w.name),
                "kernel": "%s<%d,%s>" % ("fa_bwd_kernel" if bwd else "fa_fwd_kernel", w.d,
                                         "bf16" if w.dtype == "bf16" else "fp16")}
    if bwd:  # the main backward kernel's summary (the row kernels are a few percent)
        roofline["traffic"] = profiled_traffic(w.name, "fa_bwd_kernel")

    cpu = None
    if not args.no_cpu_baseline:
        q64 = [q_h, k_h, v_h]
        n_heads = int(args.cpu_heads)
        if n_heads <= 0:  # about CPU_SAMPLE_FLOP of oracle work: whole heads
            n_heads = max(1, round(CPU_SAMPLE_FLOP / (flops / (w.B * w.H))))
        if bwd:
            tf, dt, desc = oracle_bwd_sample(w, *q64, do_h, n_heads=n_heads)
        else:
            tf, dt, desc = oracle_sample(w, *q64, n_heads=n_heads)
        cpu = {"value": tf, "unit": "TFLOPS", "cores": cpu_cores(), "kind": "oracle",
               "sample": desc, "seconds": dt}

    line = {
        "metric": METRIC_BWD if bwd else METRIC, "value": value, "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": w.dtype, "data": "synthetic",
        "config": dict(w.describe(), parallelism=f"replicas{world}" if world > 1 else "single",
                       l2=l2_note(w), **({"variant": variant} if variant else {}),
                       **({"pass": "bwd"} if bwd else {})),
        "gpu_launches": args.steps * (3 if bwd else 1),
        "host_us_per_call": host_us,
        "host_us_per_call_c_abi": c_abi_us,
        "clocks": clocks,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": e2e,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def parse_variant(text):
    """'stages=3,exp_split=4' -> {"stages": 3, "exp_split": 4} (None/'' -> {})."""
    out = {}
    for part in (text or "").split(","):
        if not part.strip():
            continue
        key, _, val = part.partition("=")
        key = key.strip()
        if key not in ("stages", "exp_split", "causal_order", "cta_pairs"):
            raise ValueError(f"unknown variant key {key!r} "
                             "(stages, exp_split, causal_order; cta_pairs with --pass bwd)")
        out[key] = int(val)
    return out


def run_sweep(args, w):
    """Time every kernel variant built for the workload's head dim and
    dtype (the default first), `args.sweep_reps` rounds with the order
    reversed every other round, each measurement after `args.sweep_idle`
    seconds idle so that all start from the same power state (30 launches
    by default: a burst below the board's power limit); print a Markdown
    table of medians."""
    import torch

    import exact_attention_forward_07_gb300 as fa

    dev = torch.device("cuda", torch.cuda.current_device())
    n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
    q, k, v = (x.to(dev) for x in make_workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    fp16 = int(w.dtype == "fp16")
    cands = [dict(stages=x["stages"], exp_split=x["exp_split"], causal_order=fa.FA_ORDER_AUTO)
             for x in fa.variants() if x["d"] == w.d and x["fp16"] == fp16 and not x["stats"]]
    if w.causal:  # the default kernel under each causal item order
        cands += [dict(cands[0], causal_order=o) for o in (-1, 0)]
    stream = torch.cuda.current_stream(dev)
    steps = args.steps or 30
    sampler = ClockSampler.for_device(dev.index)
    sampler.start()
    results = {i: [] for i in range(len(cands))}
    for rep in range(args.sweep_reps):
        order = list(range(len(cands)))
        if rep % 2:
            order.reverse()
        for i in order:
            kw = cands[i]
            time.sleep(args.sweep_idle)  # every entry starts from the same idle power state
            for _ in range(args.warmup):
                fa.fa_fwd_variant(q, k, v, o, lse, causal=w.causal, stream=stream, **kw)
            torch.cuda.synchronize(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            t0 = time.time()
            e0.record(stream)
            for _ in range(steps):
                fa.fa_fwd_variant(q, k, v, o, lse, causal=w.causal, stream=stream, **kw)
            e1.record(stream)
            torch.cuda.synchronize(dev)
            t1 = time.time()
            if fa.fa_get_status(stream) != 0:
                raise RuntimeError(f"kernel status error in variant {kw}")
            ms = e0.elapsed_time(e1) / steps
            mhz = [s[1] for s in sampler.samples if t0 <= s[0] <= t1 and s[1]]
            results[i].append((w.flops() / (ms * 1e-3) / 1e12, ms,
                               statistics.median(mhz) if mhz else None))
    sampler.stop()
    print(f"Sweep on {w.name} ({w.dtype}, {'causal' if w.causal else 'non-causal'}), "
          f"{args.sweep_reps} rounds x {steps} launches per variant, medians:\n")
    print("| stages | exp_split | causal order | TFLOPS | ms | SM MHz | FLOP/clk/SM |")
    print("|---|---|---|---|---|---|---|")
    for i, x in enumerate(cands):
        order = {fa.FA_ORDER_AUTO: "auto", -1: "heaviest first"}.get(
            x["causal_order"], f"head by head, {x['causal_order']} tail heads")
        order = order if w.causal else "-"
        tf = statistics.median(r[0] for r in results[i])
        ms = statistics.median(r[1] for r in results[i])
        clk = [r[2] for r in results[i] if r[2]]
        mhz = statistics.median(clk) if clk else None
        fpc = w.flops() / (ms * 1e-3 * mhz * 1e6 * n_sm) if mhz else None
        print(f"| {x['stages']} | {x['exp_split']} | {order} | {tf:.1f} | {ms:.4f} | "
              f"{mhz if mhz else 'n/a'} | {fpc:.0f} |" if fpc else
              f"| {x['stages']} | {x['exp_split']} | {order} | {tf:.1f} | {ms:.4f} | n/a | n/a |")
    return 0


def run_rescale_stats(args, w):
    """Run the counting build once on the workload and print how often the
    O rescale fired (JSON)."""
    import torch

    import exact_attention_forward_07_gb300 as fa

    dev = torch.device("cuda", torch.cuda.current_device())
    q, k, v = (x.to(dev) for x in make_workload_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    out = {"workload": w.name}
    for thr in (8.0, 0.0):
        stats = torch.zeros(4, dtype=torch.int64, device=dev)
        fa.fa_fwd_variant(q, k, v, o, lse, causal=w.causal, rescale_threshold=thr, stats=stats)
        torch.cuda.synchronize(dev)
        if fa.fa_get_status() != 0:
            raise RuntimeError("kernel status error in the counting build")
        need, rows, wres, wblk = (int(x) for x in stats.cpu())
        out[f"tau={thr:g}"] = {
            "row_blocks_after_first": rows, "rows_rescaled": need,
            "row_rescale_rate": need / rows if rows else None,
            "warp_blocks_after_first": wblk, "warp_blocks_rescaling": wres,
            "warp_rescale_rate": wres / wblk if wblk else None}
    print(json.dumps(out), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: about 2 s of work for our arm, 500 for the "
                         "reference arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--e2e-chunks", type=int, default=8)
    ap.add_argument("--cpu-heads", type=int, default=0,
                    help="heads in the cpu_baseline sample (0: about 1.1e12 FLOP of them)")
    ap.add_argument("--pass", dest="pass_", choices=["fwd", "bwd"], default="fwd",
                    help="time the forward (default) or the backward")
    ap.add_argument("--variant", default="",
                    help="kernel variant, e.g. stages=3,exp_split=4 (fa_fwd_variant), or "
                         "cta_pairs=1 with --pass bwd (fa_bwd_variant)")
    ap.add_argument("--sweep", action="store_true", help="time every built variant")
    ap.add_argument("--sweep-reps", type=int, default=5)
    ap.add_argument("--sweep-idle", type=float, default=0.5,
                    help="seconds idle before each sweep measurement")
    ap.add_argument("--rescale-stats", action="store_true",
                    help="count the O rescales of the workload (counting build)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    _, world, _ = dist_env()
    if world != args.gpus:
        if args.gpus != 1 or world != 1:
            print(f"note: --gpus {args.gpus} but WORLD_SIZE={world}; using WORLD_SIZE",
                  file=sys.stderr)
    w = WORKLOADS[args.workload]
    if args.sweep:
        return run_sweep(args, w)
    if args.rescale_stats:
        return run_rescale_stats(args, w)
    if args.impl == "reference":
        if args.steps is None:
            args.steps = 500
        return run_reference(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
