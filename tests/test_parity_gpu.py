"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle
on identical seeded inputs.

Bar (from the target's stated tolerances): on O, max |dO| <= 2e-2 and
mean |dO| <= 2e-3; on LSE, |dLSE| <= 1e-3 * max(1, |LSE|) (relative, with
an absolute floor of 1e-3 where LSE is near zero).

Small and medium shapes are compared element by element over the whole
output; they span several 128-row tiles, ragged tails (N % 128 != 0), an
odd number of Q tiles (the second tile of the last pair absent), N = 1 and
both head dims and dtypes, and so is the bench's workload
[8,16,4096,128] (both masks) at full size.  The other full-size workloads
are compared on sampled rows (first/last rows, tile boundaries, middle,
seeded random rows) of a spread of heads, computed by the oracle one by
one.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import WORKLOADS, make_qkv, make_workload_inputs, sample_rows
from tests.margins import record

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 2e-2, 2e-3, 1e-3


def fa():
    import exact_attention_forward_07_gb300 as m
    return m


def run_gpu(q, k, v, causal, scale=None, stream=None, rescale_threshold=None):
    dev = torch.device("cuda")
    o, lse = fa().forward(q.to(dev), k.to(dev), v.to(dev), causal=causal, scale=scale,
                          stream=stream, rescale_threshold=rescale_threshold)
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    return o.float().cpu().numpy(), lse.cpu().numpy()


def assert_close(o, lse, o_ref, lse_ref, what=""):
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    d_o = np.abs(o - o_ref)
    d_l = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    record("fwd", what, max_abs_o=d_o.max(), mean_abs_o=d_o.mean(), max_rel_lse=d_l.max())
    assert d_o.max() <= O_MAX, f"{what}: max|dO| {d_o.max():.3g}"
    assert d_o.mean() <= O_MEAN, f"{what}: mean|dO| {d_o.mean():.3g}"
    assert d_l.max() <= LSE_REL, f"{what}: max rel dLSE {d_l.max():.3g}"


SMALL = [
    # B, H, N, d, dtype
    (1, 1, 128, 64, torch.bfloat16),
    (1, 1, 1, 64, torch.bfloat16),
    (1, 1, 127, 128, torch.bfloat16),
    (1, 2, 129, 64, torch.bfloat16),
    (2, 1, 200, 128, torch.bfloat16),
    (1, 3, 384, 128, torch.bfloat16),   # 3 Q tiles: second tile of pair 1 absent
    (2, 2, 640, 64, torch.bfloat16),
    (1, 2, 1000, 128, torch.bfloat16),
    (1, 1, 333, 128, torch.float16),
    (2, 2, 512, 64, torch.float16),
    (2, 4, 1024, 128, torch.bfloat16),
    (1, 2, 2048 + 77, 128, torch.float16),
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", SMALL,
                         ids=[f"b{b}h{h}n{n}d{d}-{str(t)[6:]}" for b, h, n, d, t in SMALL])
def test_parity_full_tensor(B, H, N, d, dtype, causal):
    q, k, v = make_qkv(B, H, N, d, dtype, seed=100 + N + d)
    o, lse = run_gpu(q, k, v, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
    assert_close(o, lse, o_ref, lse_ref, f"{B},{H},{N},{d},{dtype},causal={causal}")


@pytest.mark.parametrize("name", ["tiny_b1h1n128d64", "b4h16n1024d64", "b4h16n1024d64_causal"])
def test_parity_small_workloads_full(name):
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    assert_close(o, lse, o_ref, lse_ref, name)


@pytest.mark.parametrize("name", ["b8h16n4096d128", "b8h16n4096d128_causal"])
def test_parity_bench_workload_full(name):
    """The bench's workload, both masks, element by element over the whole
    output: 524,288 rows of O and LSE against the oracle (about 1.1e12 fp64
    FLOP non-causal; seconds on the host's cores)."""
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, w.causal, w.scale)
    assert_close(o, lse, o_ref, lse_ref, name)


def spread_heads(BH, n):
    return sorted({int(x) for x in np.linspace(0, BH - 1, n)})


@pytest.mark.parametrize("name", ["b8h16n4096d128", "b8h16n4096d128_causal",
                                  "b1h32n16384d128_causal", "b16h32n8192d128_fp16_peaked"])
def test_parity_large_workloads_sampled(name):
    w = WORKLOADS[name]
    q, k, v = make_workload_inputs(w)
    o, lse = run_gpu(q, k, v, w.causal)
    BH = w.B * w.H
    heads = spread_heads(BH, 32)
    # oracle on the selected heads only (rows re-indexed into the subset)
    qs, ks, vs = (x.reshape(BH, 1, w.N, w.d)[heads].reshape(1, len(heads), w.N, w.d)
                  for x in (q, k, v))
    rows = sample_rows(1, len(heads), w.N, n_random=24, seed=7)
    o_ref, lse_ref = oracle.attn_fwd(qs, ks, vs, w.causal, w.scale, rows=rows)
    head_idx = np.asarray(heads)[rows // w.N]
    flat = head_idx * w.N + rows % w.N
    o_got = o.reshape(BH * w.N, w.d)[flat]
    lse_got = lse.reshape(-1)[flat]
    assert_close(o_got, lse_got, o_ref, lse_ref, name)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_parity_causal_head_by_head_order():
    """A causal launch whose K/V (128 MiB) outgrow L2 and whose static rounds
    balance as well head by head as heaviest-pair-first, so the library takes
    its items head by head: one seeded row of every (head, Q tile) is checked,
    so a work item that went missing or to the wrong head cannot pass."""
    B, H, N, d = 8, 64, 1024, 64
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=4242)
    o, lse = run_gpu(q, k, v, True)
    BH, tiles = B * H, N // 128
    rng = np.random.default_rng(11)
    rows = np.array([h * N + t * 128 + int(rng.integers(0, 128))
                     for h in range(BH) for t in range(tiles)], dtype=np.int64)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1.0 / math.sqrt(d), rows=rows)
    assert_close(o.reshape(BH * N, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref,
                 "causal [8,64,1024,64] head by head")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


TAIL_WINDOW_SHAPES = [(1, 32, 16384, 128), (8, 16, 4096, 128), (4, 48, 4096, 64)]


@pytest.mark.parametrize("B,H,N,d", TAIL_WINDOW_SHAPES,
                         ids=[f"b{b}h{h}n{n}d{d}" for b, h, n, d in TAIL_WINDOW_SHAPES])
def test_parity_causal_tail_window_order(B, H, N, d):
    """Causal launches taken head by head with their last heads taken
    together (the host's choice for these shapes on a 152-SM GB300): one
    seeded row of every (head, Q tile) is checked against the oracle, so a
    work item that went missing or to the wrong head cannot pass."""
    import ctypes
    f = fa().lib().fa_causal_order
    f.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int]
    f.restype = ctypes.c_int
    g = f(B, H, N, d, torch.cuda.get_device_properties(0).multi_processor_count)
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=4300 + N + H)
    o, lse = run_gpu(q, k, v, True)
    BH, tiles = B * H, N // 128
    rng = np.random.default_rng(13)
    rows = np.array([h * N + t * 128 + int(rng.integers(0, 128))
                     for h in range(BH) for t in range(tiles)], dtype=np.int64)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1.0 / math.sqrt(d), rows=rows)
    assert_close(o.reshape(BH * N, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref,
                 f"causal {B},{H},{N},{d} order {g}")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))


def test_uniform_attention_q_zero():
    """Q = 0: every visible key gets the same weight (closed form)."""
    q, k, v = make_qkv(1, 2, 300, 128, torch.bfloat16, seed=5, q_zero=True)
    for causal in (False, True):
        o, lse = run_gpu(q, k, v, causal)
        vv = v.double().numpy()
        if causal:
            want = np.cumsum(vv, axis=2) / np.arange(1, 301)[None, None, :, None]
            want_lse = np.log(np.arange(1, 301))[None, None, :].repeat(2, axis=1)
        else:
            want = np.broadcast_to(vv.mean(axis=2, keepdims=True), vv.shape)
            want_lse = np.full((1, 2, 300), math.log(300))
        assert_close(o, lse, want, want_lse, f"q=0 causal={causal}")


def test_constant_v_rows():
    q, k, v = make_qkv(2, 2, 512, 64, torch.bfloat16, seed=6, k_mult=4.0)
    u = torch.linspace(-3, 3, 64).to(torch.bfloat16)
    v = u.expand(2, 2, 512, 64).contiguous()
    for causal in (False, True):
        o, _ = run_gpu(q, k, v, causal)
        assert np.max(np.abs(o - u.float().numpy())) <= O_MAX


def test_causal_row_zero_is_v0():
    q, k, v = make_qkv(1, 4, 256, 128, torch.bfloat16, seed=8)
    o, lse = run_gpu(q, k, v, True)
    assert np.max(np.abs(o[:, :, 0] - v[:, :, 0].float().numpy())) <= 1e-2
    s00 = (q[:, :, 0].double() * k[:, :, 0].double()).sum(-1).numpy() / math.sqrt(128)
    assert np.max(np.abs(lse[:, :, 0] - s00) / np.maximum(1, np.abs(s00))) <= LSE_REL


# Non-causal shapes whose last round of work items is cut into key
# pieces (the wave-tail split): k = 4 pieces with every item split, an odd
# tile count with a ragged end, k = 3 with one block per piece, and a mix of
# whole and split items (k = 2) on a 152-SM device.
SPLIT_SHAPES = [
    (1, 2, 4096, torch.bfloat16),
    (1, 1, 4097, torch.float16),
    (1, 5, 300, torch.bfloat16),
    (1, 64, 2048, torch.bfloat16),
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("B,H,N,dtype", SPLIT_SHAPES,
                         ids=[f"b{b}h{h}n{n}-{str(t)[6:]}" for b, h, n, t in SPLIT_SHAPES])
def test_parity_wave_tail_split(B, H, N, dtype, d):
    q, k, v = make_qkv(B, H, N, d, dtype, seed=60 + N + H)
    o, lse = run_gpu(q, k, v, False)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 1.0 / math.sqrt(d))
    assert_close(o, lse, o_ref, lse_ref, f"split {B},{H},{N},d={d},{dtype}")


def _random_cases(n, seed, n_lo=1, n_hi=1500, bh_hi=(4, 5)):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        N = int(rng.integers(n_lo, n_hi))
        B = int(rng.integers(1, bh_hi[0]))
        H = int(rng.integers(1, bh_hi[1]))
        causal = bool(rng.integers(0, 2))
        dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float16
        cases.append((B, H, N, d, causal, dtype))
    return cases


RANDOM_CASES = _random_cases(32, seed=2026)
# longer sequences (more blocks per item, more phases per barrier), fewer heads
RANDOM_CASES += _random_cases(16, seed=2027, n_lo=1500, n_hi=6000, bh_hi=(3, 3))


@pytest.mark.parametrize("B,H,N,d,causal,dtype", RANDOM_CASES,
                         ids=[f"b{b}h{h}n{n}d{d}-{'c' if c else 'f'}-{str(t)[6:]}"
                              for b, h, n, d, c, t in RANDOM_CASES])
def test_parity_random_shapes(B, H, N, d, causal, dtype):
    """Seeded random shapes (any N up to 1500, both head dims, both masks,
    both dtypes; many of them hit the wave-tail split, ragged tails and odd
    tile counts), full tensors against the oracle."""
    q, k, v = make_qkv(B, H, N, d, dtype, seed=1000 + N * 7 + d + B * 3 + H)
    o, lse = run_gpu(q, k, v, causal)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
    assert_close(o, lse, o_ref, lse_ref, f"{B},{H},{N},{d},causal={causal},{dtype}")


@pytest.mark.parametrize("d", [64, 128])
def test_wave_tail_split_peaked_rows(d):
    """Pieces of one row see very different maxima (K scaled x6, sorted so
    the largest logits sit in the last piece): the merge must weigh each
    piece by its own max and sum."""
    B, H, N = 1, 3, 2048
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=61, k_mult=6.0)
    order = torch.argsort((q[0, 0].float().mean(0) @ k[0].float().transpose(-1, -2)).mean(0))
    k = k[:, :, order].contiguous()
    for thr in (0.0, 8.0):
        o, lse = run_gpu(q, k, v, False, rescale_threshold=thr)
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 1.0 / math.sqrt(d))
        assert_close(o, lse, o_ref, lse_ref, f"split peaked thr={thr} d={d}")


def test_deterministic_bitwise():
    q, k, v = make_qkv(2, 8, 1536, 128, torch.bfloat16, seed=9)
    dev = torch.device("cuda")
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    for causal in (False, True):
        o1, l1 = fa().forward(q, k, v, causal=causal)
        o2, l2 = fa().forward(q, k, v, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
    # split items: the merge reads the pieces in a fixed order, whichever
    # piece finishes last
    q, k, v = (x.to(dev) for x in make_qkv(1, 2, 4096, 128, torch.bfloat16, seed=19))
    o1, l1 = fa().forward(q, k, v, causal=False)
    for _ in range(3):
        o2, l2 = fa().forward(q, k, v, causal=False)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("B,H,N,causal", [(1, 2, 4096, False), (2, 4, 1000, True)],
                         ids=["split", "causal"])
def test_cuda_graph_capture_replays_bitwise(B, H, N, causal):
    """fa_fwd captured into a CUDA graph replays to the eager result bit for
    bit, twice: launches inside stream capture work, and the wave-tail
    split's scratch (here 128 pieces) becomes a graph allocation."""
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in make_qkv(B, H, N, 128, torch.bfloat16, seed=14))
    o_ref, l_ref = fa().forward(q, k, v, causal=causal)
    torch.cuda.synchronize()
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa().fa_fwd(q, k, v, o, lse, causal=causal)
    for _ in range(2):
        o.zero_()
        lse.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa().fa_get_status() == 0


@pytest.mark.parametrize("fn", ["fa_fwd", "fa_fwd_ex"])
def test_split_calls_after_setup_allocate_nothing(fn):
    """The caller owns every buffer and, once the device is set up (the
    first call reserves the split-scratch pool), calls issued on one stream
    allocate no device memory: in a fresh process, after a causal first
    call, ten split calls leave free device memory unchanged."""
    from tests.fresh_process import free_memory_around_split_calls
    free0, free1 = free_memory_around_split_calls(fn)
    assert free1 == free0


def test_concurrent_streams_split_scratch():
    """Calls on two streams at once, each with a split last round, take
    separate scratch from the stream-ordered pool: both match their serial
    results bit for bit."""
    dev = torch.device("cuda")
    a = [x.to(dev) for x in make_qkv(1, 2, 4096, 128, torch.bfloat16, seed=15)]
    b = [x.to(dev) for x in make_qkv(1, 3, 2048, 128, torch.bfloat16, seed=16)]
    ref_a = fa().forward(*a, causal=False)
    ref_b = fa().forward(*b, causal=False)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        with torch.cuda.stream(s1):
            oa = fa().forward(*a, causal=False, stream=s1)
        with torch.cuda.stream(s2):
            ob = fa().forward(*b, causal=False, stream=s2)
        torch.cuda.synchronize()
        assert torch.equal(oa[0], ref_a[0]) and torch.equal(oa[1], ref_a[1])
        assert torch.equal(ob[0], ref_b[0]) and torch.equal(ob[1], ref_b[1])
    assert fa().fa_get_status() == 0


def test_side_stream_and_explicit_scale():
    q, k, v = make_qkv(1, 2, 700, 64, torch.bfloat16, seed=10)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        o, lse = run_gpu(q, k, v, True, scale=0.3, stream=s)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 0.3)
    assert_close(o, lse, o_ref, lse_ref, "side stream")


def test_caller_buffers_and_no_write_on_error():
    dev = torch.device("cuda")
    q, k, v = (x.to(dev) for x in make_qkv(1, 1, 256, 64, torch.bfloat16, seed=11))
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 1, 256), 7.0, device=dev)
    rc = fa().lib().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                           lse.data_ptr(), 1, 1, 256, 64, 0, float("nan"), None)
    assert rc == fa().FA_ERR_SCALE
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)
    fa().fa_fwd(q, k, v, o, lse, causal=False)
    torch.cuda.synchronize()
    assert not torch.any(o == 7.0)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("thr", [0.0, 3.0, 8.0, 12.0])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("dtype,k_mult", [(torch.bfloat16, 1.0), (torch.float16, 4.0),
                                          (torch.bfloat16, 6.0)], ids=["bf16", "fp16x4", "bf16x6"])
def test_rescale_threshold_parity(thr, causal, dtype, k_mult, d):
    """Every rescale threshold gives the same softmax (numerator and
    denominator share the stale max), including 0 = rescale whenever the
    running max grows and peaked rows (K scaled up) that force rescales.
    Both head dims: at d=64 the rescale waits for the previous PV through
    its own barrier (P has columns apart from S there)."""
    q, k, v = make_qkv(2, 3, 1100, d, dtype, seed=31, k_mult=k_mult)
    o, lse = run_gpu(q, k, v, causal, rescale_threshold=thr)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
    assert_close(o, lse, o_ref, lse_ref, f"thr={thr} d={d}")


def test_sorted_keys_force_rescale_every_block():
    """Keys whose logits grow block after block make the running max rise on
    every block, so the O rescale runs on every block for every row."""
    B, H, N, d = 1, 2, 1024, 64
    q = torch.ones(B, H, N, d)
    k = torch.linspace(0, 3.0, N).view(1, 1, N, 1).expand(B, H, N, d).contiguous()
    _, _, v = make_qkv(B, H, N, d, torch.float32, seed=32)
    q, k, v = (x.to(torch.bfloat16) for x in (q, k, v))
    for thr in (0.0, 8.0):
        for causal in (False, True):
            o, lse = run_gpu(q, k, v, causal, rescale_threshold=thr)
            o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
            assert_close(o, lse, o_ref, lse_ref, f"sorted keys thr={thr} causal={causal}")


def test_bounded_wait_gives_up_and_context_survives():
    """Failure detection without a fault: a wait that nothing satisfies gives
    up after its limit, the status word reports FA_ERR_TIMEOUT once (then is
    cleared), and the context still runs a correct forward afterwards."""
    gave_up = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert fa().fa_get_status() == 0
    rc = fa().lib().fa_selftest_wait_timeout(20000, gave_up.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    assert gave_up.item() == 1
    assert fa().fa_get_status() == fa().FA_ERR_TIMEOUT
    assert fa().fa_get_status() == 0
    q, k, v = make_qkv(1, 2, 256, 64, torch.bfloat16, seed=12)
    o, lse = run_gpu(q, k, v, True)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, True, 1.0 / 8.0)
    assert_close(o, lse, o_ref, lse_ref, "after timeout self-test")


@pytest.mark.parametrize("chunks", [1, 3, 5, 0])
def test_fa_fwd_host_matches_oracle(chunks):
    """The pipelined host-buffer forward (fa_fwd_host: chunks of heads, copies
    and kernels on the library's three streams) gives the oracle's result,
    twice in a row (staging memory taken from the pool again)."""
    B, H, N, d = 2, 5, 333, 128
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=40)
    pin = [x.pin_memory() for x in (q, k, v)]
    for causal in (True, False):
        o = torch.empty_like(q).pin_memory()
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
        fa().fa_fwd_host(*pin, o, lse, causal=causal, chunks=chunks)
        assert fa().fa_get_status() == 0
        o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
        assert_close(o.float().numpy(), lse.numpy(), o_ref, lse_ref, f"host chunks={chunks}")


def test_fa_fwd_host_pageable_fp16_and_bitwise():
    """Pageable (not pinned) fp16 host buffers, d = 64, a chunk count above
    B*H (clamped): the same bits as fa_fwd_ex on device copies of the inputs."""
    B, H, N, d = 1, 3, 1000, 64
    q, k, v = make_qkv(B, H, N, d, torch.float16, seed=41)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32)
    fa().fa_fwd_host(q, k, v, o, lse, causal=False, chunks=7)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    od = torch.empty_like(qd)
    ld = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa().fa_fwd_ex(qd, kd, vd, od, ld, causal=False)
    torch.cuda.synchronize()
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_parity_maximum_sequence_length(causal, d):
    """N = FA_MAX_N (2^20), the longest sequence the boundary accepts: the
    index arithmetic over 8192 Q tiles and 8192 K/V blocks (and, at d=64,
    the S-free / PV-done barriers over that many phases), checked on
    sampled rows (first/last rows, tile boundaries, middle, random)."""
    N = fa().FA_MAX_N
    q, k, v = make_qkv(1, 1, N, d, torch.bfloat16, seed=50 + d)
    o, lse = run_gpu(q, k, v, causal)
    rows = sample_rows(1, 1, N, n_random=8, seed=51)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d), rows=rows)
    assert_close(o.reshape(N, d)[rows], lse.reshape(-1)[rows], o_ref, lse_ref,
                 f"N=2^20 d={d} causal={causal}")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
