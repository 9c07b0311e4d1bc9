"""fa_fwd_noalloc: the entry point whose wave-tail split scratch is a fixed
device array instead of pool memory, for callers that cannot allocate
device memory while they run (a server whose caching allocator holds the
GPU's memory, a real-time loop that must not reach the allocator).

It must give fa_fwd_ex's result bit for bit (two calls in a row, so the
second finds the array as the first left it), allocate no device memory,
and reject (without writing o or lse) a call whose split needs more than
FA_NOALLOC_SCRATCH_BYTES.  The split plans are computed from the device's
own SM count with the library's rule, so the cases test what they claim on
any GB300 partition.  This file is collected last."""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv
from tests.fresh_process import free_memory_around_split_calls

pytestmark = pytest.mark.gpu

NOALLOC_BYTES = 16 << 20


def fa():
    import exact_attention_forward_07_gb300 as m
    return m


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def split_plan(B, H, N, d, causal, G):
    """(pieces, scratch bytes) of the library's wave-tail split on G SMs:
    the last round's R = items mod G items, when R <= G / 2, are cut into
    k = min(G // R, 4, Q tiles) pieces.  (0, 0) when nothing is split."""
    tiles = (N + 127) // 128
    items = B * H * ((tiles + 1) // 2)
    R = items % G
    if causal or R == 0:
        return 0, 0
    k = min(G // R, 4, tiles)
    if k < 2:
        return 0, 0
    pieces = R * k
    st = (pieces * 256 * 3 * 4 + 255) // 256 * 256
    return pieces, pieces * 256 * d * 4 + st + R * 4


def _raw(fn, q, k, v, o, lse, causal, thr=8.0):
    B, H, N, d = q.shape
    return getattr(fa().lib(), fn)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, int(causal), 1.0 / math.sqrt(d),
                                   int(q.dtype == torch.float16), thr, None)


def _inputs(B, H, N, d, dtype, seed):
    return [x.cuda() for x in make_qkv(B, H, N, d, dtype, seed=seed)]


# (B, H, N, d, dtype, causal): calls whose split fits the array on a 152-SM
# GB300 (68, 30, 112 and 128 pieces) and a call that needs no scratch
ACCEPTED = [
    (1, 1, 4097, 128, torch.float16, False),
    (1, 5, 300, 128, torch.bfloat16, False),
    (1, 64, 2048, 128, torch.bfloat16, False),
    (1, 2, 4096, 128, torch.bfloat16, True),
    (2, 4, 1024, 64, torch.bfloat16, False),
]


@pytest.mark.parametrize("B,H,N,d,dtype,causal", ACCEPTED,
                         ids=[f"b{b}h{h}n{n}d{d}-{str(t)[6:]}-{'causal' if c else 'full'}"
                              for b, h, n, d, t, c in ACCEPTED])
def test_noalloc_bitwise_equals_fa_fwd_ex(B, H, N, d, dtype, causal):
    pieces, need = split_plan(B, H, N, d, causal, sm_count())
    if need > NOALLOC_BYTES:
        pytest.skip(f"on {sm_count()} SMs this split needs {need} bytes: rejected by design")
    q, k, v = _inputs(B, H, N, d, dtype, seed=70 + N)
    o1 = torch.empty_like(q)
    l1 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    assert _raw("fa_fwd_ex", q, k, v, o1, l1, causal) == 0
    for _ in range(2):  # the second call finds the array as the first left it
        o2 = torch.full_like(q, 3.0)
        l2 = torch.full_like(l1, 3.0)
        assert _raw("fa_fwd_noalloc", q, k, v, o2, l2, causal) == 0
        torch.cuda.synchronize()
        assert fa().fa_get_status() == 0
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_accepted_cases_exercise_the_split():
    """On a 152-SM GB300 the non-causal accepted cases really split (else
    the bitwise test above would only cover whole items)."""
    G = sm_count()
    plans = [split_plan(B, H, N, d, c, G)[0] for B, H, N, d, _, c in ACCEPTED if not c]
    if G == 152:
        assert plans == [68, 30, 112, 128]
    assert any(p > 0 for p in plans) or G != 152


def test_noalloc_matches_oracle():
    B, H, N, d = 1, 5, 300, 128
    q, k, v = make_qkv(B, H, N, d, torch.bfloat16, seed=71)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = torch.empty_like(qd)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa().fa_fwd_noalloc(qd, kd, vd, o, lse)
    o_ref, lse_ref = oracle.attn_fwd(q, k, v, False, 1.0 / math.sqrt(d))
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    assert np.abs(o - o_ref).max() <= 2e-2 and np.abs(o - o_ref).mean() <= 2e-3
    assert (np.abs(lse - lse_ref) / np.maximum(1.0, np.abs(lse_ref))).max() <= 1e-3


def _oversize_shape(G):
    """A non-causal d = 128 shape whose split does not fit the array on G
    SMs ([1,2,4096,128] on 152: 128 pieces, 17.2 MB), or None."""
    for H in range(1, 65):
        if split_plan(1, H, 4096, 128, False, G)[1] > NOALLOC_BYTES:
            return 1, H, 4096, 128
    return None


def test_noalloc_rejects_oversize_without_writing():
    """A split that does not fit is rejected before any launch; fa_fwd_ex
    serves the same call, and its causal form (no split) is accepted."""
    shape = _oversize_shape(sm_count())
    if shape is None:
        pytest.skip(f"no N=4096 d=128 split exceeds the array on {sm_count()} SMs")
    B, H, N, d = shape
    q, k, v = _inputs(B, H, N, d, torch.bfloat16, seed=72)
    o = torch.full_like(q, 7.0)
    lse = torch.full((B, H, N), 7.0, device="cuda")
    assert _raw("fa_fwd_noalloc", q, k, v, o, lse, False) == fa().FA_ERR_SCRATCH
    torch.cuda.synchronize()
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)
    with pytest.raises(fa().FaError) as err:
        fa().fa_fwd_noalloc(q, k, v, o, lse)
    assert err.value.code == fa().FA_ERR_SCRATCH
    assert "FA_NOALLOC_SCRATCH_BYTES" in fa().fa_strerror(fa().FA_ERR_SCRATCH)
    assert _raw("fa_fwd_ex", q, k, v, o, lse, False) == 0
    assert _raw("fa_fwd_noalloc", q, k, v, o, lse, True) == 0
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    assert not torch.any(lse == 7.0)


def test_noalloc_allocates_no_device_memory():
    """Fresh process: after a scratch-free first call, ten split calls of
    fa_fwd_noalloc leave free device memory unchanged."""
    if split_plan(1, 64, 2048, 128, False, sm_count())[0] == 0:
        pytest.skip("[1,64,2048,128] does not split on this SM count")
    free0, free1 = free_memory_around_split_calls("fa_fwd_noalloc")
    assert free1 == free0
