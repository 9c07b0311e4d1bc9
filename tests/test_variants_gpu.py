"""The library's kernel variants (fa_fwd_variant: K/V ring depth, a share
of the softmax's exponentials on the FMA pipes, rescale counters) compute
the same attention as the default: each is compared with the oracle on
shapes with several tiles, ragged tails and both masks, at the target's
tolerances.  The counting build gives the default's bits and exact totals.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv
from tests.margins import record

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_REL = 2e-2, 2e-3, 1e-3


def fa():
    import exact_attention_forward_07_gb300 as m
    return m


def _variants():
    import exact_attention_forward_07_gb300 as m
    try:
        return [v for v in m.variants() if not v["stats"]]
    except Exception:  # library not built on this machine: collected, skipped
        return []


VARIANTS = _variants()
SHAPES = [(2, 3, 1000, False), (1, 2, 1100, True), (1, 64, 2048, False), (2, 2, 333, True)]


def _check(o, lse, o_ref, lse_ref, what):
    d_o = np.abs(o - o_ref)
    d_l = np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse)), what
    record("variant", what, max_abs_o=d_o.max(), mean_abs_o=d_o.mean(), max_rel_lse=d_l.max())
    assert d_o.max() <= O_MAX and d_o.mean() <= O_MEAN and d_l.max() <= LSE_REL, (
        f"{what}: max|dO| {d_o.max():.3g} mean|dO| {d_o.mean():.3g} rel dLSE {d_l.max():.3g}")


@pytest.mark.parametrize("B,H,N,causal", SHAPES,
                         ids=[f"b{b}h{h}n{n}-{'c' if c else 'f'}" for b, h, n, c in SHAPES])
@pytest.mark.parametrize("var", VARIANTS,
                         ids=[f"d{v['d']}-{'fp16' if v['fp16'] else 'bf16'}-s{v['stages']}"
                              f"-x{v['exp_split']}" for v in VARIANTS])
def test_variant_parity(var, B, H, N, causal):
    d = var["d"]
    dtype = torch.float16 if var["fp16"] else torch.bfloat16
    k_mult = 4.0 if var["fp16"] else 1.0
    q, k, v = make_qkv(B, H, N, d, dtype, seed=500 + N + H, k_mult=k_mult)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fa().fa_fwd_variant(qd, kd, vd, o, lse, causal=causal, stages=var["stages"],
                        exp_split=var["exp_split"])
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, causal, 1.0 / math.sqrt(d))
    _check(o.float().cpu().numpy(), lse.cpu().numpy(), o_ref, lse_ref, str(var))


@pytest.mark.parametrize("d,dtype", [(64, torch.bfloat16), (128, torch.bfloat16),
                                     (128, torch.float16)], ids=["d64-bf16", "d128-bf16",
                                                                 "d128-fp16"])
def test_counting_build_bitwise_and_totals(d, dtype):
    """Causal [2,3,1000,d]: Q tile t has t+1 K/V blocks, so the counters of
    (row, block) pairs and of warp-blocks after each tile's first block are
    known exactly; with keys sorted so that every block raises the running
    max and tau = 0, every such row rescales.  The outputs equal the
    default build's bit for bit."""
    B, H, N = 2, 3, 1000
    T = (N + 127) // 128
    q, k, v = make_qkv(B, H, N, d, dtype, seed=77)
    dev = torch.device("cuda")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    o1, o2 = torch.empty_like(qd), torch.empty_like(qd)
    l1 = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    l2 = torch.empty_like(l1)
    stats = torch.zeros(4, dtype=torch.int64, device=dev)
    fa().fa_fwd_ex(qd, kd, vd, o1, l1, causal=True)
    fa().fa_fwd_variant(qd, kd, vd, o2, l2, causal=True, stats=stats)
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    after_first = B * H * sum(range(T))  # tile t: t blocks after its first
    need, rows, wres, wblk = (int(x) for x in stats.cpu())
    assert rows == 128 * after_first and wblk == 8 * after_first
    assert 0 <= need <= rows and 0 <= wres <= wblk
    # every block raises every row's max: Q = 1, and keys constant within a
    # 128-key block and 0.25 larger in each block (exact in 16 bits), so
    # each block's scores exceed the previous block's by 0.25 * sqrt(d);
    # N a multiple of 128, so no row lies past the end
    N2 = 1024
    T2 = N2 // 128
    qs = torch.ones(B, H, N2, d)
    ks = (torch.arange(N2) // 128 * 0.25).view(1, 1, N2, 1).expand(B, H, N2, d).contiguous()
    vs = make_qkv(B, H, N2, d, dtype, seed=78)[2].to(dev)
    qs, ks = qs.to(dtype).to(dev), ks.to(dtype).to(dev)
    o3 = torch.empty_like(vs)
    l3 = torch.empty((B, H, N2), dtype=torch.float32, device=dev)
    stats.zero_()
    fa().fa_fwd_variant(qs, ks, vs, o3, l3, causal=True, rescale_threshold=0.0, stats=stats)
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    need, rows, wres, wblk = (int(x) for x in stats.cpu())
    after_first2 = B * H * sum(range(T2))
    assert rows == 128 * after_first2 and need == rows and wres == wblk == 8 * after_first2
