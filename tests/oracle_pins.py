"""Checks that pin the CPU oracle to facts fixed by the pages and by the
mathematics of softmax, independently of the oracle's own code.

Each check takes an oracle library handle (`lib`, None = the default build)
so that the mutation tests can run the same checks against deliberately
broken builds of the oracle source and see at least one of them fail.

Sources of each fact:
 - rows of P sum to one, masked entries are zero, constant V gives that
   constant: properties of the softmax-weighted average that the exact
   attention of the pages computes ("flash attention v2 论文" search page:
   the output equals conventional attention).
 - online tiling == 3-pass softmax for any split: the online-softmax
   recurrence of the FlashAttention v2 diagram ("online_softmax_update") and
   the v4 Blackwell diagram's pseudo-code panel (m_new = max(m, rowmax),
   rescale acc and l by exp(m - m_new), P = exp(S - m_new), acc += P V,
   final O = acc / l), with l also gaining rowsum(P) each tile.
 - two-tile hand derivation: the practice panel of both diagrams, item 1.
 - Q = 0, N = 1, key shift, key/value permutation: closed forms and
   invariants of softmax.
 - decimal brute force: the definition in 50-digit decimal arithmetic.
"""
from __future__ import annotations

import math
import os
from decimal import Decimal, getcontext

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def rand_qkv(B, H, N, d, seed, k_mult=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, N, d)) * k_mult
    v = rng.standard_normal((B, H, N, d))
    return q, k, v


def online_softmax_reference(q, k, v, causal, scale, bc):
    """The pages' online-softmax recurrence, written independently of the
    oracle: sweep key tiles of width `bc`, keep running (m, l, acc)."""
    B, H, N, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros(q.shape[:3])
    for b in range(B):
        for h in range(H):
            for i in range(N):
                m, l, acc = -math.inf, 0.0, np.zeros(d)
                last = i if causal else N - 1
                for j0 in range(0, last + 1, bc):
                    j1 = min(j0 + bc, last + 1)
                    s = scale * (k[b, h, j0:j1] @ q[b, h, i])
                    m_new = max(m, float(s.max()))
                    alpha = math.exp(m - m_new) if m != -math.inf else 0.0
                    p = np.exp(s - m_new)
                    acc = acc * alpha + p @ v[b, h, j0:j1]
                    l = l * alpha + float(p.sum())
                    m = m_new
                o[b, h, i] = acc / l
                lse[b, h, i] = m + math.log(l)
    return o, lse


def check_probs_sum_to_one(lib=None):
    for causal in (False, True):
        q, k, _ = rand_qkv(2, 2, 19, 8, 11)
        p = oracle.attn_probs(q, k, causal, 0.37, lib=lib)
        assert np.all(np.abs(p.sum(-1) - 1.0) <= 1e-12)
        assert np.all(p >= 0)


def check_masked_entries_zero(lib=None):
    q, k, _ = rand_qkv(1, 2, 23, 8, 12)
    p = oracle.attn_probs(q, k, True, 0.5, lib=lib)
    upper = np.triu(np.ones((23, 23), dtype=bool), 1)
    assert np.all(p[..., upper] == 0.0)
    assert np.all(p[..., ~upper] > 0.0)
    p_full = oracle.attn_probs(q, k, False, 0.5, lib=lib)
    assert np.all(p_full > 0.0)


def check_online_tiling_matches(lib=None):
    q, k, v = rand_qkv(1, 2, 29, 5, 13, k_mult=3.0)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.61, lib=lib)
        for bc in (1, 2, 3, 7, 16, 29):
            o_on, lse_on = online_softmax_reference(q, k, v, causal, 0.61, bc)
            assert np.max(np.abs(o - o_on)) <= 1e-12, (causal, bc)
            assert np.max(np.abs(lse - lse_on)) <= 1e-12, (causal, bc)


def check_constant_v(lib=None):
    q, k, _ = rand_qkv(2, 1, 17, 6, 14, k_mult=2.0)
    u = np.array([0.5, -1.25, 3.0, 7.0, -0.125, 2.5])
    v = np.broadcast_to(u, q.shape).copy()
    for causal in (False, True):
        o, _ = oracle.attn_fwd(q, k, v, causal, 0.8, lib=lib)
        assert np.max(np.abs(o - u)) <= 1e-12


def check_q_zero_uniform(lib=None):
    _, k, v = rand_qkv(2, 2, 13, 4, 15)
    q = np.zeros_like(k)
    o, lse = oracle.attn_fwd(q, k, v, False, 0.9, lib=lib)
    assert np.max(np.abs(o - v.mean(axis=2, keepdims=True))) <= 1e-12
    assert np.max(np.abs(lse - math.log(13))) <= 1e-12
    o, lse = oracle.attn_fwd(q, k, v, True, 0.9, lib=lib)
    counts = np.arange(1, 14)[None, None, :, None]
    assert np.max(np.abs(o - np.cumsum(v, axis=2) / counts)) <= 1e-12
    assert np.max(np.abs(lse - np.log(np.arange(1, 14))[None, None, :])) <= 1e-12


def check_single_key(lib=None):
    q, k, v = rand_qkv(3, 2, 1, 7, 16)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.7, lib=lib)
        assert np.max(np.abs(o - v)) <= 1e-12
        want = 0.7 * np.sum(q * k, axis=-1)
        assert np.max(np.abs(lse - want)) <= 1e-12


def load_two_tile_golden():
    vals = {}
    with open(os.path.join(GOLDEN, "two_tile_online_softmax.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *nums = line.split()
            vals[key] = np.array([float(x) for x in nums])
    return vals


def check_two_tile_golden(lib=None):
    g = load_two_tile_golden()
    q = g["q"].reshape(1, 1, 2, 1)
    k = g["k"].reshape(1, 1, 2, 1)
    v = g["v"].reshape(1, 1, 2, 1)
    o, lse = oracle.attn_fwd(q, k, v, False, 1.0, lib=lib)
    assert np.max(np.abs(o.reshape(-1) - g["o_noncausal"])) <= 1e-12
    assert np.max(np.abs(lse.reshape(-1) - g["lse_noncausal"])) <= 1e-12
    o, lse = oracle.attn_fwd(q, k, v, True, 1.0, lib=lib)
    assert np.max(np.abs(o.reshape(-1) - g["o_causal"])) <= 1e-12
    assert np.max(np.abs(lse.reshape(-1) - g["lse_causal"])) <= 1e-12


def check_key_shift(lib=None):
    q, k, v = rand_qkv(1, 2, 21, 6, 17)
    u = np.array([0.3, -0.2, 1.1, 0.0, -0.7, 0.25])
    for causal in (False, True):
        o0, lse0 = oracle.attn_fwd(q, k, v, causal, 0.45, lib=lib)
        o1, lse1 = oracle.attn_fwd(q, k + u, v, causal, 0.45, lib=lib)
        assert np.max(np.abs(o1 - o0)) <= 1e-12
        assert np.max(np.abs(lse1 - (lse0 + 0.45 * (q @ u)))) <= 1e-12


def check_permutation(lib=None):
    q, k, v = rand_qkv(2, 1, 25, 5, 18, k_mult=2.0)
    perm = np.random.default_rng(3).permutation(25)
    o0, lse0 = oracle.attn_fwd(q, k, v, False, 0.55, lib=lib)
    o1, lse1 = oracle.attn_fwd(q, k[:, :, perm], v[:, :, perm], False, 0.55, lib=lib)
    assert np.max(np.abs(o1 - o0)) <= 1e-12
    assert np.max(np.abs(lse1 - lse0)) <= 1e-12


def check_torch_softmax(lib=None):
    import torch
    q, k, v = rand_qkv(2, 3, 40, 16, 19, k_mult=1.5)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.25, lib=lib)
        qt, kt, vt = (torch.from_numpy(x) for x in (q, k, v))
        s = 0.25 * qt @ kt.transpose(-1, -2)
        if causal:
            mask = torch.triu(torch.ones(40, 40, dtype=torch.bool), 1)
            s = s.masked_fill(mask, float("-inf"))
        want_p = torch.softmax(s, dim=-1)
        want_o = want_p @ vt
        want_lse = torch.logsumexp(s, dim=-1)
        e_o = np.max(np.abs(o - want_o.numpy()))
        e_l = np.max(np.abs(lse - want_lse.numpy()))
        p = oracle.attn_probs(q, k, causal, 0.25, lib=lib)
        e_p = np.max(np.abs(p - want_p.numpy()))
        assert e_o <= 1e-12 and e_l <= 1e-12 and e_p <= 1e-14, (causal, e_o, e_l, e_p)


def decimal_row(q, k, v, b, h, i, causal, scale, digits=50):
    getcontext().prec = digits
    D = Decimal
    sc = D(repr(scale))
    last = i if causal else q.shape[2] - 1
    s = []
    for j in range(last + 1):
        dot = sum(D(repr(float(a))) * D(repr(float(c)))
                  for a, c in zip(q[b, h, i], k[b, h, j]))
        s.append(sc * dot)
    m = max(s)
    w = [(x - m).exp() for x in s]
    l = sum(w)
    o = [sum(w[j] * D(repr(float(v[b, h, j, c]))) for j in range(last + 1)) / l
         for c in range(q.shape[3])]
    lse = m + l.ln()
    return np.array([float(x) for x in o]), float(lse)


def check_decimal_bruteforce(lib=None):
    q, k, v = rand_qkv(1, 2, 33, 6, 20, k_mult=4.0)
    for causal in (False, True):
        o, lse = oracle.attn_fwd(q, k, v, causal, 0.35, lib=lib)
        for (h, i) in ((0, 0), (0, 17), (1, 32), (1, 5)):
            want_o, want_lse = decimal_row(q, k, v, 0, h, i, causal, 0.35)
            assert np.max(np.abs(o[0, h, i] - want_o)) <= 1e-13
            assert abs(lse[0, h, i] - want_lse) <= 1e-13


ALL_CHECKS = [
    check_probs_sum_to_one,
    check_masked_entries_zero,
    check_online_tiling_matches,
    check_constant_v,
    check_q_zero_uniform,
    check_single_key,
    check_two_tile_golden,
    check_key_shift,
    check_permutation,
    check_torch_softmax,
    check_decimal_bruteforce,
]
