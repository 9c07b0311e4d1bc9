"""GPU parity of the backward (fa_bwd, through the C ABI) against the fp64
CPU oracle on identical seeded inputs.

The GPU backward takes the GPU forward's O and LSE (as a caller would) and
an output gradient dO ~ N(0,1); the oracle differentiates the definition
from Q, K, V and dO alone.  The target states tolerances for the forward
only; the bar here follows from the arithmetic: the kernel rounds P and dS
to the 16-bit input type for its tensor-core products and the outputs to
16 bits, each a relative error of at most 2^-9 (bf16) whose contributions
average out over the sums, and D = rowsum(dO * O) uses the rounded O.  So
per gradient tensor G: ||dG||_F <= 1e-2 ||G||_F (five times one bf16
rounding) and max |dG| <= 2e-2 max |G|, with ||G||_F and max |G| floored at
1e-3 sqrt(size) and 1e-3 (the gradients of these N(0,1) inputs are of order
0.1 to 1; the floor only matters where the exact gradient is zero, e.g. dQ
and dK with a single key).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv
from tests.margins import record

pytestmark = pytest.mark.gpu

REL_FRO, REL_MAX = 1e-2, 2e-2


def fa():
    import exact_attention_forward_07_gb300 as m
    return m


def grad_inputs(B, H, N, d, dtype, seed, k_mult=1.0):
    q, k, v = make_qkv(B, H, N, d, dtype, seed=seed, k_mult=k_mult)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 3)
    do = torch.randn((B, H, N, d), generator=g, dtype=torch.float32).to(dtype)
    return q, k, v, do


def run_gpu_bwd(q, k, v, do, causal, scale=None, cta_pairs=None):
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa().forward(qd, kd, vd, causal=causal, scale=scale)
    dq, dk, dv = fa().backward(qd, kd, vd, o, lse, dod, causal=causal, scale=scale,
                               cta_pairs=cta_pairs)
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    return [x.float().cpu().numpy() for x in (dq, dk, dv)]


def assert_grads_close(got, ref, what):
    for name, g, r in zip(("dQ", "dK", "dV"), got, ref):
        assert np.all(np.isfinite(g)), f"{what} {name}: non-finite"
        err = g - r
        fro = np.linalg.norm(err) / max(np.linalg.norm(r), 1e-3 * math.sqrt(r.size))
        mx = np.abs(err).max() / max(np.abs(r).max(), 1e-3)
        record("bwd", f"{what} {name}", rel_fro=fro, rel_max=mx)
        assert fro <= REL_FRO and mx <= REL_MAX, f"{what} {name}: rel Fro {fro:.3g}, rel max {mx:.3g}"


SMALL = [
    (1, 1, 128, 64, torch.bfloat16),
    (1, 1, 1, 64, torch.bfloat16),
    (1, 2, 200, 128, torch.bfloat16),
    (2, 2, 333, 64, torch.float16),
    (1, 3, 384, 128, torch.bfloat16),
    (2, 1, 1000, 128, torch.float16),
    (1, 2, 2048 + 77, 128, torch.bfloat16),
    (2, 2, 1024, 64, torch.bfloat16),
    # d = 64 walks its three-stage Q/dO ring: two steps (fewer than the
    # stages), and six with a ragged tail (the ring wraps twice)
    (1, 1, 200, 64, torch.bfloat16),
    (1, 2, 5 * 128 + 19, 64, torch.float16),
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", SMALL,
                         ids=[f"b{b}h{h}n{n}d{d}-{str(t)[6:]}" for b, h, n, d, t in SMALL])
def test_bwd_parity_full_tensor(B, H, N, d, dtype, causal):
    q, k, v, do = grad_inputs(B, H, N, d, dtype, seed=800 + N + d)
    got = run_gpu_bwd(q, k, v, do, causal)
    ref = oracle.attn_bwd(q, k, v, do, causal, 1.0 / math.sqrt(d))
    assert_grads_close(got, ref, f"{B},{H},{N},{d},{dtype},causal={causal}")


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_parity_bench_shape_heads(causal):
    """[8,16,4096,128] bf16, the forward's gate shape: the whole launch on
    the GPU, three spread heads (every row of them) against the oracle."""
    B, H, N, d = 8, 16, 4096, 128
    q, k, v, do = grad_inputs(B, H, N, d, torch.bfloat16, seed=900)
    got = run_gpu_bwd(q, k, v, do, causal)
    heads = [0, 61, 127]
    sub = [x.reshape(B * H, 1, N, d)[heads].reshape(1, len(heads), N, d) for x in (q, k, v, do)]
    ref = oracle.attn_bwd(*sub, causal, 1.0 / math.sqrt(d))
    got = [g.reshape(B * H, N, d)[heads].reshape(1, len(heads), N, d) for g in got]
    assert_grads_close(got, ref, f"[8,16,4096,128] causal={causal}")


def test_bwd_peaked_rows_fp16():
    """K scaled x4 (the peaked fp16 workload's values): P close to one-hot."""
    q, k, v, do = grad_inputs(1, 2, 1024, 128, torch.float16, seed=901, k_mult=4.0)
    for causal in (False, True):
        got = run_gpu_bwd(q, k, v, do, causal)
        ref = oracle.attn_bwd(q, k, v, do, causal, 1.0 / math.sqrt(128))
        assert_grads_close(got, ref, f"peaked causal={causal}")


def test_bwd_closed_forms():
    """One key: dV = dO and dQ = dK = 0.  Constant V rows: dQ = dK = 0."""
    q, k, v, do = grad_inputs(2, 3, 1, 64, torch.bfloat16, seed=902)
    dq, dk, dv = run_gpu_bwd(q, k, v, do, False)
    assert np.max(np.abs(dv - do.float().numpy())) <= 1e-2
    # dS = P (dO.v - D): D is the same dot product summed in another order
    assert np.max(np.abs(dq)) <= 1e-3 and np.max(np.abs(dk)) <= 1e-3
    q, k, _, do = grad_inputs(1, 2, 300, 128, torch.bfloat16, seed=903)
    v = torch.linspace(-2, 2, 128).to(torch.bfloat16).expand(1, 2, 300, 128).contiguous()
    for causal in (False, True):
        dq, dk, _ = run_gpu_bwd(q, k, v, do, causal)
        # dS = P (dO.v - dO.o) with o = v up to O's rounding: tiny, not exact
        assert np.max(np.abs(dq)) <= 2e-2 and np.max(np.abs(dk)) <= 2e-2


def test_bwd_dk_dv_bitwise_repeatable():
    """dK and dV come from a fixed order of MMAs: bitwise the same on a
    second run.  dQ is added up with atomics in any order: close."""
    q, k, v, do = grad_inputs(2, 4, 1536, 128, torch.bfloat16, seed=904)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    for causal in (False, True):
        o, lse = fa().forward(qd, kd, vd, causal=causal)
        a = fa().backward(qd, kd, vd, o, lse, dod, causal=causal)
        b = fa().backward(qd, kd, vd, o, lse, dod, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])
        assert torch.allclose(a[0].float(), b[0].float(), rtol=1e-2, atol=1e-3)
    assert fa().fa_get_status() == 0


def test_bwd_reused_workspace_and_side_stream():
    """A workspace left dirty by one call serves the next (nothing needs to
    be cleared); calls on a side stream."""
    q, k, v, do = grad_inputs(1, 2, 700, 64, torch.bfloat16, seed=905)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    ws = torch.full((fa().fa_bwd_workspace_size(1, 2, 700, 64),), 0x7F, dtype=torch.uint8,
                    device=dev)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    ref = oracle.attn_bwd(q, k, v, do, True, 0.3)
    with torch.cuda.stream(s):
        o, lse = fa().forward(qd, kd, vd, causal=True, scale=0.3, stream=s)
        for _ in range(2):
            dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
            fa().fa_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, causal=True, scale=0.3, stream=s)
            s.synchronize()
            assert_grads_close([x.float().cpu().numpy() for x in (dq, dk, dv)], ref, "reuse")
    assert fa().fa_get_status() == 0


def test_bwd_cuda_graph_capture_replays():
    """fa_bwd allocates nothing and runs on the caller's stream, so it can be
    captured into a CUDA graph: replays give the eager dK and dV bit for bit
    and dQ up to the order of its additions."""
    q, k, v, do = grad_inputs(1, 3, 1000, 128, torch.bfloat16, seed=906)
    dev = torch.device("cuda")
    qd, kd, vd, dod = (x.to(dev) for x in (q, k, v, do))
    o, lse = fa().forward(qd, kd, vd, causal=True)
    ref = fa().backward(qd, kd, vd, o, lse, dod, causal=True)
    dq, dk, dv = (torch.empty_like(qd) for _ in range(3))
    ws = torch.empty(fa().fa_bwd_workspace_size(1, 3, 1000, 128), dtype=torch.uint8, device=dev)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa().fa_bwd(qd, kd, vd, o, lse, dod, dq, dk, dv, ws, causal=True)
    for _ in range(2):
        for x in (dq, dk, dv):
            x.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
        assert torch.allclose(dq.float(), ref[0].float(), rtol=1e-2, atol=1e-3)
    assert fa().fa_get_status() == 0


def _random_bwd_cases(n, seed, n_lo=1, n_hi=1500):
    rng = np.random.default_rng(seed)
    cases = []
    for _ in range(n):
        d = int(rng.choice([64, 128]))
        N = int(rng.integers(n_lo, n_hi))
        B = int(rng.integers(1, 3))
        H = int(rng.integers(1, 4))
        causal = bool(rng.integers(0, 2))
        dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float16
        cases.append((B, H, N, d, causal, dtype))
    return cases


RANDOM_BWD = _random_bwd_cases(16, seed=3030)


@pytest.mark.parametrize("B,H,N,d,causal,dtype", RANDOM_BWD,
                         ids=[f"b{b}h{h}n{n}d{d}-{'c' if c else 'f'}-{str(t)[6:]}"
                              for b, h, n, d, c, t in RANDOM_BWD])
def test_bwd_parity_random_shapes(B, H, N, d, causal, dtype):
    """Seeded random shapes: any N up to 1500 (ragged last tiles, a single
    partial tile), both head dims, masks and dtypes, full tensors."""
    q, k, v, do = grad_inputs(B, H, N, d, dtype, seed=7000 + N + d + H)
    got = run_gpu_bwd(q, k, v, do, causal)
    ref = oracle.attn_bwd(q, k, v, do, causal, 1.0 / math.sqrt(d))
    assert_grads_close(got, ref, f"{B},{H},{N},{d},causal={causal},{dtype}")


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_parity_long_sequence(causal, d):
    """N = 8192 (64 key blocks per query block, 64 query blocks per key
    block: the dQ accumulators take 64 additions per element), two heads,
    every row against the oracle."""
    q, k, v, do = grad_inputs(1, 2, 8192, d, torch.bfloat16, seed=7100 + d)
    got = run_gpu_bwd(q, k, v, do, causal)
    ref = oracle.attn_bwd(q, k, v, do, causal, 1.0 / math.sqrt(d))
    assert_grads_close(got, ref, f"[1,2,8192,{d}] causal={causal}")


def _check_sampled(q, k, v, do, got, causal, rows, what):
    """dQ on sampled rows against the oracle, and the identities that hold at
    any size: sum_j dV_j = sum_i dO_i (rows of P sum to one) and
    sum_j dK_j = 0 (rows of dS sum to zero), per head and column.

    dV and dK accumulate in tensor memory over every query block, 8 MMA
    steps each, and the tensor core's fp32 accumulation does not round to
    nearest: the sums drift low by up to 2^-23 per step, coherently across
    keys (measured: 1.2e-3 at N = 2^20, 65536 steps; 3e-5 at N = 2^14).  The
    bound on the dV identity is that drift plus 1e-3 for the 16-bit
    roundings; dK's sum cancels and keeps the plain 1e-3."""
    B, H, N, d = q.shape
    dq, dk, dv = got
    ref_dq = oracle.attn_bwd_dq_rows(q, k, v, do, causal, 1.0 / math.sqrt(d), rows)
    assert_grads_close([dq.reshape(-1, d)[rows]], [ref_dq], f"{what} sampled rows")
    do64 = do.double().numpy().reshape(B * H, N, d)
    dv64 = dv.astype(np.float64).reshape(B * H, N, d)
    dk64 = dk.astype(np.float64).reshape(B * H, N, d)
    steps = (N + 127) // 128 * 8
    tol_v = steps * 2.0 ** -23 + 1e-3
    err_v = np.abs(dv64.sum(1) - do64.sum(1)) / (np.abs(dv64).sum(1) + 1e-3)
    err_k = np.abs(dk64.sum(1)) / (np.abs(dk64).sum(1) + 1e-6)
    record("bwd", f"{what} dV-sum identity", rel=err_v.max(), bound=tol_v)
    record("bwd", f"{what} dK-sum identity", rel=err_k.max(), bound=1e-3)
    assert err_v.max() <= tol_v, (what, err_v.max(), tol_v)
    assert err_k.max() <= 1e-3, (what, err_k.max())


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_maximum_sequence_length_sampled(causal, d):
    """N = FA_MAX_N (2^20), one head: 8192 key blocks, each walking up to
    8192 query blocks (the dQ accumulators take up to 8192 additions per
    element); sampled dQ rows against the oracle, the dK and dV sums at full
    size."""
    N = fa().FA_MAX_N
    q, k, v, do = grad_inputs(1, 1, N, d, torch.bfloat16, seed=7200 + d)
    got = run_gpu_bwd(q, k, v, do, causal)
    rows = sample_rows_bwd(1, 1, N, n_random=6, seed=73)
    _check_sampled(q, k, v, do, got, causal, rows, f"N=2^20 d={d} causal={causal}")


def test_bwd_long_causal_workload_sampled():
    """The long causal workload [1,32,16384,128] (the forward's default bench
    shape): sampled dQ rows of eight spread heads, the sums at full size."""
    from attn_inputs import WORKLOADS, make_workload_inputs
    w = WORKLOADS["b1h32n16384d128_causal"]
    q, k, v = make_workload_inputs(w)
    g = torch.Generator(device="cpu")
    g.manual_seed(74)
    do = torch.randn(q.shape, generator=g).to(q.dtype)
    got = run_gpu_bwd(q, k, v, do, True)
    rows = sample_rows_bwd(1, 32, w.N, n_random=3, seed=75, heads=range(0, 32, 4))
    _check_sampled(q, k, v, do, got, True, rows, w.name)


def sample_rows_bwd(B, H, N, n_random, seed, heads=None):
    from attn_inputs import sample_rows
    return sample_rows(B, H, N, n_random=n_random, seed=seed, heads=heads)


# Shapes for the kernel that runs CTAs in clusters of two (fa_bwd_variant,
# cta_pairs = 1): one key block (a working CTA and an idle one), two (one
# pair), three (a pair and a lone block), ragged and longer sequences.
PAIR_SHAPES = [
    (1, 1, 1, 64, torch.bfloat16),
    (1, 2, 100, 128, torch.bfloat16),
    (1, 2, 256, 128, torch.bfloat16),
    (1, 2, 384, 64, torch.float16),
    (2, 3, 1000, 128, torch.bfloat16),
    (1, 2, 2048 + 77, 128, torch.bfloat16),
    (2, 2, 1024, 64, torch.bfloat16),
    (1, 1, 4096, 128, torch.float16),
]


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
@pytest.mark.parametrize("B,H,N,d,dtype", PAIR_SHAPES,
                         ids=[f"b{b}h{h}n{n}d{d}-{str(t)[6:]}" for b, h, n, d, t in PAIR_SHAPES])
def test_bwd_cta_pairs_parity(B, H, N, d, dtype, causal):
    """The paired kernel against the oracle, and against the one-CTA kernel:
    dK and dV come from the same MMAs in the same order (bitwise equal);
    dQ only groups its fp32 additions differently."""
    q, k, v, do = grad_inputs(B, H, N, d, dtype, seed=1700 + N + d)
    got = run_gpu_bwd(q, k, v, do, causal, cta_pairs=1)
    ref = oracle.attn_bwd(q, k, v, do, causal, 1.0 / math.sqrt(d))
    assert_grads_close(got, ref, f"pairs {B},{H},{N},{d},{dtype},causal={causal}")
    single = run_gpu_bwd(q, k, v, do, causal, cta_pairs=0)
    assert np.array_equal(got[1], single[1]) and np.array_equal(got[2], single[2])
    scale_q = max(np.abs(single[0]).max(), 1e-3)
    assert np.abs(got[0] - single[0]).max() <= 2.0 ** -7 * scale_q


@pytest.mark.parametrize("causal", [False, True], ids=["full", "causal"])
def test_bwd_cta_pairs_bench_shape_heads(causal):
    """[8,16,4096,128] bf16 through the paired kernel, three heads against
    the oracle."""
    B, H, N, d = 8, 16, 4096, 128
    q, k, v, do = grad_inputs(B, H, N, d, torch.bfloat16, seed=900)
    got = run_gpu_bwd(q, k, v, do, causal, cta_pairs=1)
    heads = [0, 61, 127]
    sub = [x.reshape(B * H, 1, N, d)[heads].reshape(1, len(heads), N, d) for x in (q, k, v, do)]
    ref = oracle.attn_bwd(*sub, causal, 1.0 / math.sqrt(d))
    got = [g.reshape(B * H, N, d)[heads].reshape(1, len(heads), N, d) for g in got]
    assert_grads_close(got, ref, f"pairs [8,16,4096,128] causal={causal}")
