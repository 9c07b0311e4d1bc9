"""Checks that pin the backward CPU oracle (oracle.attn_bwd) to facts that
do not come from its own code.

The gradients are those of L = sum(dO * O) with O the attention forward.
Each check takes an oracle library handle (`lib`, None = the default build)
for the backward, so the mutation tests can run the same checks against
deliberately broken builds of attn_bwd_oracle.c; the forward always comes
from the default build, which is pinned on its own (tests/oracle_pins.py).

Sources of each fact:
 - central finite differences of the forward oracle: the definition of a
   derivative (and the "backward idea" of the FlashAttention v4 Blackwell
   pipeline diagram's pseudo-code panel: the backward pass differentiates
   the same forward);
 - constant V rows: O no longer depends on Q or K, so dQ = dK = 0;
 - one key: O = v_0 whatever Q and K are, so dV = dO and dQ = dK = 0;
 - Q = 0: uniform weights 1/|A(i)|, dK = 0 and closed forms for dV, dQ;
 - rows of the softmax Jacobian sum to zero, so sum_j dK_j = 0;
 - adding a vector to every key leaves O, hence every gradient, unchanged;
 - linearity of the gradients in dO;
 - torch autograd of a library softmax in fp64 (a special case that
   reduces to a library routine);
 - a two-query, two-key case derived by hand (tests/golden/two_key_backward.txt).
"""
from __future__ import annotations

import numpy as np

import oracle
from tests.oracle_pins import rand_qkv

TOL = 1e-12


def _grads(q, k, v, do, causal, scale, lib):
    return oracle.attn_bwd(q, k, v, do, causal, scale, lib=lib)


def check_finite_differences(lib=None):
    """Every entry of dQ, dK, dV of a small case against central differences
    of L = sum(dO * O) computed with the forward oracle."""
    q, k, v = rand_qkv(1, 2, 6, 3, 31, k_mult=1.5)
    do = np.random.default_rng(32).standard_normal(q.shape)
    h = 1e-6
    for causal in (False, True):
        grads = _grads(q, k, v, do, causal, 0.83, lib)

        def loss(qq, kk, vv):
            o, _ = oracle.attn_fwd(qq, kk, vv, causal, 0.83)
            return float(np.sum(do * o))
        for which, g in enumerate(grads):
            fd = np.zeros_like(g)
            for idx in np.ndindex(*g.shape):
                args = [q.copy(), k.copy(), v.copy()]
                args[which][idx] += h
                up = loss(*args)
                args[which][idx] -= 2 * h
                dn = loss(*args)
                fd[idx] = (up - dn) / (2 * h)
            assert np.max(np.abs(g - fd)) <= 1e-7, (causal, "qkv"[which], np.max(np.abs(g - fd)))


def check_constant_v(lib=None):
    q, k, _ = rand_qkv(2, 1, 9, 4, 33, k_mult=2.0)
    v = np.broadcast_to(np.array([0.5, -1.0, 2.0, 0.25]), q.shape).copy()
    do = np.random.default_rng(34).standard_normal(q.shape)
    for causal in (False, True):
        dq, dk, _ = _grads(q, k, v, do, causal, 0.6, lib)
        assert np.max(np.abs(dq)) <= TOL and np.max(np.abs(dk)) <= TOL


def check_single_key(lib=None):
    q, k, v = rand_qkv(2, 2, 1, 5, 35)
    do = np.random.default_rng(36).standard_normal(q.shape)
    for causal in (False, True):
        dq, dk, dv = _grads(q, k, v, do, causal, 0.9, lib)
        assert np.max(np.abs(dv - do)) <= TOL
        assert np.max(np.abs(dq)) <= TOL and np.max(np.abs(dk)) <= TOL


def check_q_zero_closed_form(lib=None):
    """Q = 0: p_ij = 1/n_i over the n_i visible keys.  Then
    dV_j = sum_{i sees j} dO_i / n_i, dK = 0, and
    dQ_i = scale / n_i * sum_{j visible} (dO_i.v_j - mean_k dO_i.v_k) k_j."""
    _, k, v = rand_qkv(1, 2, 7, 3, 37)
    q = np.zeros_like(k)
    do = np.random.default_rng(38).standard_normal(q.shape)
    scale = 0.7
    for causal in (False, True):
        dq, dk, dv = _grads(q, k, v, do, causal, scale, lib)
        N = q.shape[2]
        want_dv = np.zeros_like(v)
        want_dq = np.zeros_like(q)
        for h in range(2):
            for i in range(N):
                vis = list(range(i + 1)) if causal else list(range(N))
                n = len(vis)
                dp = np.array([do[0, h, i] @ v[0, h, j] for j in vis])
                for t, j in enumerate(vis):
                    want_dv[0, h, j] += do[0, h, i] / n
                    want_dq[0, h, i] += scale / n * (dp[t] - dp.mean()) * k[0, h, j]
        assert np.max(np.abs(dk)) <= TOL
        assert np.max(np.abs(dv - want_dv)) <= TOL
        assert np.max(np.abs(dq - want_dq)) <= TOL


def check_dk_sums_to_zero(lib=None):
    q, k, v = rand_qkv(2, 2, 11, 4, 39, k_mult=2.5)
    do = np.random.default_rng(40).standard_normal(q.shape)
    for causal in (False, True):
        _, dk, _ = _grads(q, k, v, do, causal, 0.5, lib)
        assert np.max(np.abs(dk.sum(axis=2))) <= 1e-11


def check_key_shift_invariance(lib=None):
    q, k, v = rand_qkv(1, 2, 10, 4, 41)
    do = np.random.default_rng(42).standard_normal(q.shape)
    u = np.array([0.4, -0.3, 1.2, -0.8])
    for causal in (False, True):
        g0 = _grads(q, k, v, do, causal, 0.65, lib)
        g1 = _grads(q, k + u, v, do, causal, 0.65, lib)
        for a, b in zip(g0, g1):
            assert np.max(np.abs(a - b)) <= 1e-11


def check_linear_in_dout(lib=None):
    q, k, v = rand_qkv(1, 1, 8, 3, 43)
    rng = np.random.default_rng(44)
    d1, d2 = rng.standard_normal(q.shape), rng.standard_normal(q.shape)
    for causal in (False, True):
        g1 = _grads(q, k, v, d1, causal, 0.75, lib)
        g2 = _grads(q, k, v, d2, causal, 0.75, lib)
        g12 = _grads(q, k, v, d1 + 2.0 * d2, causal, 0.75, lib)
        for a, b, c in zip(g1, g2, g12):
            assert np.max(np.abs(c - (a + 2.0 * b))) <= 1e-11


def check_torch_autograd(lib=None):
    import torch
    q, k, v = rand_qkv(2, 2, 24, 8, 45, k_mult=1.5)
    do = np.random.default_rng(46).standard_normal(q.shape)
    for causal in (False, True):
        dq, dk, dv = _grads(q, k, v, do, causal, 0.35, lib)
        qt, kt, vt = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        s = 0.35 * qt @ kt.transpose(-1, -2)
        if causal:
            mask = torch.triu(torch.ones(24, 24, dtype=torch.bool), 1)
            s = s.masked_fill(mask, float("-inf"))
        o = torch.softmax(s, dim=-1) @ vt
        o.backward(torch.from_numpy(do))
        for ours, ref in ((dq, qt.grad), (dk, kt.grad), (dv, vt.grad)):
            assert np.max(np.abs(ours - ref.numpy())) <= 1e-12


def check_two_key_golden(lib=None):
    """The hand derivation of tests/golden/two_key_backward.txt (two
    queries, two keys, d = 1), both masks."""
    import os
    vals = {}
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                           "two_key_backward.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *nums = line.split()
                vals[key] = np.array([float(x) for x in nums])
    q, k, v, do = (vals[n].reshape(1, 1, 2, 1) for n in ("q", "k", "v", "dout"))
    for causal, tag in ((False, "noncausal"), (True, "causal")):
        dq, dk, dv = _grads(q, k, v, do, causal, 1.0, lib)
        assert np.max(np.abs(dq.reshape(-1) - vals["dq_" + tag])) <= TOL, (tag, dq)
        assert np.max(np.abs(dk.reshape(-1) - vals["dk_" + tag])) <= TOL, (tag, dk)
        assert np.max(np.abs(dv.reshape(-1) - vals["dv_" + tag])) <= TOL, (tag, dv)


def check_dq_rows_finite_differences(lib=None):
    """The row-sampled dQ against central differences of the forward
    oracle's L = sum(dO * O), for a few rows of a small case (both masks)."""
    q, k, v = rand_qkv(1, 2, 7, 3, 47, k_mult=1.5)
    do = np.random.default_rng(48).standard_normal(q.shape)
    rows = np.array([0, 3, 6, 7, 13])
    h = 1e-6
    for causal in (False, True):
        got = oracle.attn_bwd_dq_rows(q, k, v, do, causal, 0.7, rows, lib=lib)

        def loss(qq):
            o, _ = oracle.attn_fwd(qq, k, v, causal, 0.7)
            return float(np.sum(do * o))
        for r, flat in enumerate(rows):
            bh, i = divmod(int(flat), 7)
            for c in range(3):
                qp, qm = q.copy(), q.copy()
                qp[0, bh, i, c] += h
                qm[0, bh, i, c] -= h
                fd = (loss(qp) - loss(qm)) / (2 * h)
                assert abs(got[r, c] - fd) <= 1e-7, (causal, flat, c, got[r, c], fd)


ALL_CHECKS = [check_dq_rows_finite_differences, check_two_key_golden, check_finite_differences, check_constant_v, check_single_key,
              check_q_zero_closed_form, check_dk_sums_to_zero, check_key_shift_invariance,
              check_linear_in_dout, check_torch_autograd]
