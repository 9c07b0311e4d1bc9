"""Pins of the CPU oracle (no GPU): each check compares it with a fact that
does not come from the oracle itself (see tests/oracle_pins.py)."""
import numpy as np
import pytest

import oracle
from tests import oracle_pins as pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


def test_rows_subset_matches_full_and_thread_count():
    q, k, v = pins.rand_qkv(2, 3, 37, 8, 21)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.3, nthreads=1)
        o4, lse4 = oracle.attn_fwd(q, k, v, causal, 0.3, nthreads=4)
        assert np.array_equal(o, o4) and np.array_equal(lse, lse4)
        rows = np.array([0, 5, 36, 37, 100, 2 * 3 * 37 - 1])
        ro, rl = oracle.attn_fwd(q, k, v, causal, 0.3, rows=rows, nthreads=3)
        assert np.array_equal(ro, o.reshape(-1, 8)[rows])
        assert np.array_equal(rl, lse.reshape(-1)[rows])


def test_bad_arguments():
    q, k, v = pins.rand_qkv(1, 1, 4, 2, 22)
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, k[:, :, :3], v, False, 1.0)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, k, v, False, 1.0, rows=[4])
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, k, v, False, 1.0, rows=[-1])


def test_accepts_16bit_torch_inputs_exactly():
    import torch
    from attn_inputs import make_qkv
    q, k, v = make_qkv(1, 2, 9, 4, torch.bfloat16, seed=5)
    o_t, lse_t = oracle.attn_fwd(q, k, v, True, 0.5)
    o_n, lse_n = oracle.attn_fwd(q.double().numpy(), k.double().numpy(),
                                 v.double().numpy(), True, 0.5)
    assert np.array_equal(o_t, o_n) and np.array_equal(lse_t, lse_n)
