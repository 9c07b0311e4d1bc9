"""fa_fwd_noalloc: the entry point whose wave-tail split scratch is a fixed
device array instead of pool memory.  It must give fa_fwd_ex's result
bit for bit, allocate no device memory, and reject (without writing o or
lse) a call whose split needs more than FA_NOALLOC_SCRATCH_BYTES."""
import math

import numpy as np
import pytest
import torch

import oracle
from attn_inputs import make_qkv

pytestmark = pytest.mark.gpu


def fa():
    import exact_attention_forward_07_gb300 as m
    return m


def _raw(fn, q, k, v, o, lse, causal, thr=8.0):
    B, H, N, d = q.shape
    return getattr(fa().lib(), fn)(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                   lse.data_ptr(), B, H, N, d, int(causal), 1.0 / math.sqrt(d),
                                   int(q.dtype == torch.float16), thr, None)


def _inputs(B, H, N, d, dtype, seed):
    return [x.cuda() for x in make_qkv(B, H, N, d, dtype, seed=seed)]


# (B, H, N, d, dtype, causal): split plans that fit the array (68, 30 and 112
# pieces of 134,144 bytes, 128 pieces of 68,608 bytes at d = 64, on 152 SMs)
# and a call that needs no scratch (causal)
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
    q, k, v = _inputs(B, H, N, d, dtype, seed=70 + N)
    o1, o2 = torch.empty_like(q), torch.empty_like(q)
    l1 = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    l2 = torch.empty_like(l1)
    assert _raw("fa_fwd_ex", q, k, v, o1, l1, causal) == 0
    assert _raw("fa_fwd_noalloc", q, k, v, o2, l2, causal) == 0
    torch.cuda.synchronize()
    assert fa().fa_get_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


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


def test_noalloc_rejects_oversize_without_writing():
    """[1,2,4096,128] non-causal: 32 items become 128 pieces, 17.2 MB of
    scratch > FA_NOALLOC_SCRATCH_BYTES.  Rejected before any launch;
    fa_fwd_ex serves the same call, and the causal form (no split) is
    accepted by fa_fwd_noalloc."""
    q, k, v = _inputs(1, 2, 4096, 128, torch.bfloat16, seed=72)
    o = torch.full_like(q, 7.0)
    lse = torch.full((1, 2, 4096), 7.0, device="cuda")
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
    """Free device memory is the same before and after a run of split calls
    (the first call, which loads the module and its fixed array, is made
    before the measurement)."""
    q, k, v = _inputs(1, 64, 2048, 128, torch.bfloat16, seed=73)
    o = torch.empty_like(q)
    lse = torch.empty((1, 64, 2048), dtype=torch.float32, device="cuda")
    assert _raw("fa_fwd_noalloc", q, k, v, o, lse, False) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(10):
        assert _raw("fa_fwd_noalloc", q, k, v, o, lse, False) == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert fa().fa_get_status() == 0
