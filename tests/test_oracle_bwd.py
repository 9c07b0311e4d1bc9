"""Pins of the backward CPU oracle (no GPU), and planted mistakes in copies
of its C source, each of which at least one pin must catch.  The mistakes
are planted on the CPU, in the oracle (never in the GPU path)."""
import os
import subprocess

import numpy as np
import pytest

import oracle
from tests import oracle_bwd_pins as pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "attn_bwd_oracle.c")


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check()


def test_thread_count_does_not_change_the_result():
    q, k, v = pins.rand_qkv(2, 3, 13, 4, 50)
    do = np.random.default_rng(51).standard_normal(q.shape)
    for causal in (False, True):
        a = oracle.attn_bwd(q, k, v, do, causal, 0.4, nthreads=1)
        b = oracle.attn_bwd(q, k, v, do, causal, 0.4, nthreads=5)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


def test_dq_rows_match_the_full_backward():
    """The row-sampled dQ equals the full backward oracle's dQ on the same
    rows (both masks, rows in any order, repeated rows), and rejects rows
    out of range."""
    q, k, v = pins.rand_qkv(2, 3, 19, 5, 53, k_mult=2.0)
    do = np.random.default_rng(54).standard_normal(q.shape)
    rows = np.array([0, 18, 19, 57, 113, 5, 5, 2 * 3 * 19 - 1])
    for causal in (False, True):
        dq, _, _ = oracle.attn_bwd(q, k, v, do, causal, 0.45)
        got = oracle.attn_bwd_dq_rows(q, k, v, do, causal, 0.45, rows, nthreads=3)
        assert np.max(np.abs(got - dq.reshape(-1, 5)[rows])) <= 1e-12
    with pytest.raises(RuntimeError):
        oracle.attn_bwd_dq_rows(q, k, v, do, False, 0.45, [2 * 3 * 19])


def test_bad_arguments():
    q, k, v = pins.rand_qkv(1, 1, 4, 2, 52)
    with pytest.raises(ValueError):
        oracle.attn_bwd(q, k, v, q[:, :, :3], False, 1.0)


MUTANTS = [
    ("r_dropped", "const double ds = p[j] * (dp[j] - r);", "const double ds = p[j] * dp[j];"),
    ("ds_without_p", "const double ds = p[j] * (dp[j] - r);", "const double ds = dp[j] - r;"),
    ("dq_scale_dropped", "dqi[c] += jb->scale * ds * K[j * d + c];",
     "dqi[c] += ds * K[j * d + c];"),
    ("dk_uses_key", "dK[j * d + c] += jb->scale * ds * qi[c];",
     "dK[j * d + c] += jb->scale * ds * K[j * d + c];"),
    ("dv_uses_dp", "dV[j * d + c] += p[j] * doi[c];", "dV[j * d + c] += dp[j] * doi[c];"),
    ("dp_from_query", "dot += doi[c] * V[j * d + c];", "dot += doi[c] * V[i * d + c];"),
    ("causal_off_by_one", "jb->causal ? i + 1 : N;", "jb->causal ? (i > 0 ? i : 1) : N;"),
    ("p_not_normalised", "p[j] = exp(s[j] - m) / l;", "p[j] = exp(s[j] - m);"),
    ("softmax_scale_dropped", "s[j] = jb->scale * dot;", "s[j] = dot;"),
    ("dv_not_reset", "memset(dV, 0, sizeof(double) * (size_t)(N * d));", ""),
    ("rows_r_dropped", "const double ds = exp(s[j] - m) / l * (dp[j] - rr);",
     "const double ds = exp(s[j] - m) / l * dp[j];"),
    ("rows_scale_dropped", "out[c] += jb->scale * ds * K[j * d + c];",
     "out[c] += ds * K[j * d + c];"),
]


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(tmp_path, name, find, repl):
    src = open(SRC).read()
    assert find in src, f"mutation site for {name} no longer in the oracle source"
    c_path = tmp_path / f"{name}.c"
    so_path = tmp_path / f"{name}.so"
    c_path.write_text(src.replace(find, repl, 1))
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c99", "-o", str(so_path),
                    str(c_path), "-lm", "-lpthread"], check=True)
    lib = oracle.load_library(str(so_path))
    failures = []
    for check in pins.ALL_CHECKS:
        try:
            check(lib=lib)
        except (AssertionError, RuntimeError, ValueError, FloatingPointError):
            failures.append(check.__name__)
    assert failures, f"no pin caught the planted mistake {name}"
