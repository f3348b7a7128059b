"""Pins of the CPU oracle against facts fixed by the KDA page and by mathematics.

Page: "Kimi K3: KDA, attention residuals and Stable LatentMoE" (hs-black.github.io),
Sec. 2.1 (recurrence, chunked form), Sec. 2.2 (bounded gate, 16-token
sub-chunks, e^80 bound), Sec. 2.3 (output gate), Sec. 10.2 (KCP pairs),
Sec. 13.1 (prefix cache: states restorable at block boundaries), Kimi
Linear's unbounded gate printed beside K3's in Sec. 2.2, and the ShortConv +
Swish prologue of Sec. 2.1.

Each pin is chosen so that a plausible slip in the oracle (a dropped decay, a
sign, a transposed readout, a wrong index) fails at least one of them; the
mutation tests at the end plant such slips in a copy of the oracle and check
that the pins catch them.
"""
import json
import math
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import chunked

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand(T, H, d, seed, z_std=2.0, A_std=0.5):
    r = np.random.default_rng(seed)
    q = _unit(r.standard_normal((T, H, d)))
    k = _unit(r.standard_normal((T, H, d)))
    v = r.standard_normal((T, H, d))
    z = z_std * r.standard_normal((T, H, d))
    beta = 1 / (1 + np.exp(-r.standard_normal((T, H))))
    A = A_std * r.standard_normal(H)
    return q, k, v, z, beta, A


# --------------------------------------------------------------------------
# 1. Brute force: exact rational evaluation of the page's matrix statement
#    S_t = (I - beta k k^T) Diag(alpha) S_{t-1} + beta k v^T,  o_t = S_t^T q_t
# --------------------------------------------------------------------------

def _brute(q, k, v, alpha, beta, S0):
    d = len(q[0])
    S = [[Fraction(x) for x in row] for row in S0]
    outs = []
    for t in range(len(q)):
        M = [[(Fraction(int(i == j)) - beta[t] * k[t][i] * k[t][j]) * alpha[t][j]
              for j in range(d)] for i in range(d)]
        S = [[sum(M[i][m] * S[m][j] for m in range(d)) + beta[t] * k[t][i] * v[t][j]
              for j in range(d)] for i in range(d)]
        outs.append([sum(S[i][j] * q[t][i] for i in range(d)) for j in range(d)])
    return outs, S


@pytest.mark.parametrize("T,d", [(1, 2), (3, 3), (4, 4), (4, 2)])
def test_brute_force_rational(T, d):
    r = np.random.default_rng(100 + 10 * T + d)
    dy = lambda shape: r.integers(-8, 9, size=shape) / 8.0          # dyadic, exact in fp64
    q, k, v = dy((T, 1, d)), dy((T, 1, d)), dy((T, 1, d))
    beta = r.integers(1, 8, size=(T, 1)) / 8.0
    z = r.standard_normal((T, 1, d))
    A = np.array([0.25])
    S0 = dy((1, 1, d, d))
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    g = oracle.log_decay(z[:, 0], A[0])
    alpha = [[Fraction(math.exp(x)) for x in row] for row in g]
    F = lambda a: [[Fraction(float(x)) for x in row] for row in a]
    bo, bS = _brute(F(q[:, 0]), F(k[:, 0]), F(v[:, 0]), alpha,
                    [Fraction(float(b)) for b in beta[:, 0]], F(S0[0, 0]))
    np.testing.assert_allclose(o[:, 0], np.array(bo, dtype=np.float64), rtol=0, atol=1e-12)
    np.testing.assert_allclose(S_T[0, 0], np.array(bS, dtype=np.float64), rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# 2. The chunked form of Sec. 2.1 equals the recurrence (FP64)
# --------------------------------------------------------------------------

@pytest.mark.parametrize("T,C,sub", [(64, 64, None), (64, 64, 16), (150, 64, 16),
                                     (150, 16, None), (37, 64, 16), (200, 64, None)])
def test_chunked_equals_recurrence(T, C, sub):
    q, k, v, z, beta, A = _rand(T, 2, 8, seed=T + C)
    S0 = 0.1 * np.random.default_rng(7).standard_normal((1, 2, 8, 8))
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    for h in range(2):
        g = oracle.log_decay(z[:, h], A[h])
        O, S, _ = chunked.chunked_prefill(q[:, h], k[:, h], v[:, h], g, beta[:, h], S0[0, h],
                                          C=C, sub=sub)
        np.testing.assert_allclose(O, o[:, h], rtol=0, atol=1e-12 * np.abs(o[:, h]).max())
        np.testing.assert_allclose(S, S_T[0, h], rtol=0, atol=1e-12 * np.abs(S_T[0, h]).max())


# --------------------------------------------------------------------------
# 3. Delta-rule invariant: beta = 1, |k| = 1  =>  S_t^T k_t = v_t
# --------------------------------------------------------------------------

def test_delta_invariant():
    q, k, v, z, beta, A = _rand(6, 1, 16, seed=3)
    beta[:] = 1.0
    S0 = np.random.default_rng(4).standard_normal((1, 1, 16, 16))
    for T in range(1, 7):
        _, S_T, _ = oracle.prefill(q[:T], k[:T], v[:T], z[:T], beta[:T], A, S0=S0, qk_l2norm=False)
        np.testing.assert_allclose(S_T[0, 0].T @ k[T - 1, 0], v[T - 1, 0], atol=1e-12)


# --------------------------------------------------------------------------
# 4./5. Identity (beta = 0, alpha = 1) and decay-only closed form (beta = 0)
# --------------------------------------------------------------------------

def test_identity_when_no_write_and_no_decay():
    q, k, v, z, beta, A = _rand(20, 2, 8, seed=5)
    beta[:] = 0.0
    z[:] = -1e4                      # Sigmoid -> 0, g -> 0, alpha = 1 exactly
    A[:] = 0.0
    S0 = np.random.default_rng(6).standard_normal((1, 2, 8, 8))
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    assert np.array_equal(S_T, S0)
    np.testing.assert_allclose(o[:, 0], q[:, 0] @ S0[0, 0], atol=1e-13)


def test_decay_only_closed_form():
    q, k, v, z, beta, A = _rand(30, 1, 8, seed=8)
    beta[:] = 0.0
    S0 = np.random.default_rng(9).standard_normal((1, 1, 8, 8))
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    G = np.cumsum(oracle.log_decay(z[:, 0], A[0]), axis=0)
    np.testing.assert_allclose(S_T[0, 0], np.exp(G[-1])[:, None] * S0[0, 0], rtol=1e-12)
    for t in (0, 10, 29):
        St = np.exp(G[t])[:, None] * S0[0, 0]
        np.testing.assert_allclose(o[t, 0], St.T @ q[t, 0], rtol=1e-11, atol=1e-14)


# --------------------------------------------------------------------------
# 6. Single token from the zero state:  S = beta k v^T,  o = beta (k.q) v
# --------------------------------------------------------------------------

def test_single_token_from_zero():
    q, k, v, z, beta, A = _rand(1, 3, 16, seed=10)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, qk_l2norm=False)
    for h in range(3):
        np.testing.assert_allclose(S_T[0, h], beta[0, h] * np.outer(k[0, h], v[0, h]), atol=1e-15)
        np.testing.assert_allclose(o[0, h], beta[0, h] * (k[0, h] @ q[0, h]) * v[0, h], atol=1e-14)


# --------------------------------------------------------------------------
# 7. Orthonormal keys, beta = 1, alpha = 1: every (k_i, v_i) is retrievable
# --------------------------------------------------------------------------

def test_orthonormal_key_memory():
    d = 8
    Q = np.linalg.qr(np.random.default_rng(11).standard_normal((d, d)))[0]
    k = Q.T[:, None, :]                                   # d orthonormal keys
    v = np.random.default_rng(12).standard_normal((d, 1, d))
    q = k.copy()
    z = np.full((d, 1, d), -1e4)
    beta = np.ones((d, 1))
    _, S_T, _ = oracle.prefill(q, k, v, z, beta, np.zeros(1), qk_l2norm=False)
    for i in range(d):
        np.testing.assert_allclose(S_T[0, 0].T @ k[i, 0], v[i, 0], atol=1e-12)


# --------------------------------------------------------------------------
# 8. Split invariance: prefill(T1) then prefill(T2 | S_T1) == prefill(T1+T2);
#    a decode step continues a prefill exactly
# --------------------------------------------------------------------------

def test_split_invariance_and_decode_continuation():
    q, k, v, z, beta, A = _rand(90, 2, 16, seed=13)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A)
    o1, S1, _ = oracle.prefill(q[:57], k[:57], v[:57], z[:57], beta[:57], A)
    o2, S2, _ = oracle.prefill(q[57:], k[57:], v[57:], z[57:], beta[57:], A, S0=S1)
    assert np.array_equal(np.concatenate([o1, o2]), o) and np.array_equal(S2, S_T)
    od, Sd, _ = oracle.decode_step(q[89:90], k[89:90], v[89:90], z[89:90], beta[89:90], A,
                                   oracle.prefill(q[:89], k[:89], v[:89], z[:89], beta[:89], A)[1])
    assert np.array_equal(od[0], o[89]) and np.array_equal(Sd, S_T)


def test_varlen_packing_equals_separate_calls():
    q, k, v, z, beta, A = _rand(100, 2, 8, seed=14)
    cu = np.array([0, 0, 37, 38, 100], dtype=np.int32)      # empty and 1-token sequences
    S0 = np.random.default_rng(15).standard_normal((4, 2, 8, 8))
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=S0)
    for n in range(4):
        s, e = cu[n], cu[n + 1]
        on, Sn, _ = oracle.prefill(q[s:e], k[s:e], v[s:e], z[s:e], beta[s:e], A, S0=S0[n:n + 1])
        assert np.array_equal(o[s:e], on) and np.array_equal(S_T[n], Sn[0])


# --------------------------------------------------------------------------
# 9. KCP pairs (Sec. 10.2): S_exit = M S_entry + S~, associative combine
# --------------------------------------------------------------------------

def test_kcp_pairs_and_associativity():
    q, k, v, z, beta, A = _rand(48, 1, 6, seed=16)
    g = oracle.log_decay(z[:, 0], A[0])
    S0 = np.random.default_rng(17).standard_normal((1, 1, 6, 6))
    _, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    segs = [(0, 10), (10, 31), (31, 48)]
    pairs = [chunked.kcp_pair(k[s:e, 0], v[s:e, 0], g[s:e], beta[s:e, 0]) for s, e in segs]
    left = chunked.kcp_combine(pairs[2], chunked.kcp_combine(pairs[1], pairs[0]))
    right = chunked.kcp_combine(chunked.kcp_combine(pairs[2], pairs[1]), pairs[0])
    np.testing.assert_allclose(left[0], right[0], atol=1e-13)
    np.testing.assert_allclose(left[1], right[1], atol=1e-13)
    np.testing.assert_allclose(left[0] @ S0[0, 0] + left[1], S_T[0, 0], atol=1e-12)


# --------------------------------------------------------------------------
# 10. d_v column permutation equivariance (values, outputs, states, gate)
# --------------------------------------------------------------------------

def test_value_permutation_equivariance():
    q, k, v, z, beta, A = _rand(40, 2, 8, seed=18)
    S0 = np.random.default_rng(19).standard_normal((1, 2, 8, 8))
    g_in = np.random.default_rng(20).standard_normal((40, 2, 8))
    w = np.random.default_rng(21).random(8) + 0.5
    p = np.random.default_rng(22).permutation(8)
    o, S, y = oracle.prefill(q, k, v, z, beta, A, S0=S0, g_in=g_in, norm_w=w)
    op, Sp, yp = oracle.prefill(q, k, v[..., p], z, beta, A, S0=S0[..., p], g_in=g_in[..., p],
                                norm_w=w[p])
    np.testing.assert_allclose(op, o[..., p], atol=1e-13)
    np.testing.assert_allclose(Sp, S[..., p], atol=1e-13)
    np.testing.assert_allclose(yp, y[..., p], atol=1e-13)


# --------------------------------------------------------------------------
# 11./12. Gate: range, printed values, the e^80 sub-chunk bound (golden)
# --------------------------------------------------------------------------

def test_gate_printed_values_and_range():
    gold = json.load(open(os.path.join(GOLD, "gate_bounds.json")))
    g_min = gold["g_min"]
    a_min = math.exp(oracle.log_decay(np.array([1e4]), 0.0, g_min)[0])
    assert a_min == pytest.approx(gold["min_retention"]["value"], rel=gold["min_retention"]["rel_tol"])
    z = np.linspace(-10, 10, 601)          # away from fp64 saturation of the logistic
    al = np.exp(oracle.log_decay(z, 0.3, g_min))
    assert np.all(al > math.exp(g_min)) and np.all(al < 1.0)
    four = math.exp(4 * oracle.log_decay(np.array([1e4]), 0.0, g_min)[0])
    assert four == pytest.approx(gold["four_steps_at_bound"]["value"], rel=gold["four_steps_at_bound"]["rel_tol"])
    bf16_max = (2 - 2 ** -7) * 2.0 ** 127
    assert bf16_max == pytest.approx(gold["bf16_max"]["value"], rel=gold["bf16_max"]["rel_tol"])
    assert math.log(bf16_max) == pytest.approx(gold["bf16_max"]["log_value"], abs=gold["bf16_max"]["log_tol"])


def test_gate_closed_forms():
    # Sigmoid(0) = 1/2 -> g = g_min / 2;  A_h scales the logit by e^A
    assert oracle.log_decay(np.array([0.0]), 1.7)[0] == pytest.approx(-2.5, abs=1e-15)
    x = 0.8
    assert oracle.log_decay(np.array([x]), math.log(3.0))[0] == pytest.approx(
        -5.0 / (1.0 + math.exp(-3.0 * x)), rel=1e-14)
    assert oracle.log_decay(np.array([-1e4]), 0.0)[0] == 0.0


def test_subchunk_bound_e80():
    gold = json.load(open(os.path.join(GOLD, "gate_bounds.json")))
    T, d = 64, 4
    q, k, v, _, beta, _ = _rand(T, 1, d, seed=23)
    g = np.full((T, d), gold["g_min"])                  # every step at the bound
    _, _, f_sub = chunked.chunked_prefill(q[:, 0], k[:, 0], v[:, 0], g, beta[:, 0],
                                          np.zeros((d, d)), C=64, sub=gold["subchunk_len"])
    bound = math.exp(-gold["g_min"] * gold["subchunk_len"])
    assert f_sub == pytest.approx(bound, rel=1e-12)
    assert math.log(f_sub) == pytest.approx(-gold["subchunk_log_decay_range"]["lo"], abs=1e-9)
    assert f_sub < (2 - 2 ** -7) * 2.0 ** 127            # finite in bf16 (and fp32)
    _, _, f_chunk = chunked.chunked_prefill(q[:, 0], k[:, 0], v[:, 0], g, beta[:, 0],
                                            np.zeros((d, d)), C=64, sub=None)
    assert f_chunk > 3.4e38                               # a whole 64-chunk would overflow


# --------------------------------------------------------------------------
# Output gate and L2 norm closed forms (Sec. 2.3, Sec. 2.1)
# --------------------------------------------------------------------------

def test_gate_norm_closed_forms():
    o = np.array([[3.0, 4.0]])
    y = oracle.gate_norm(o, np.zeros_like(o), eps=0.0)
    rms = math.sqrt(12.5)
    np.testing.assert_allclose(y, 0.5 * o / rms, rtol=1e-15)
    y2 = oracle.gate_norm(np.full((1, 8), -2.0), np.full((1, 8), 1e4), norm_w=np.arange(8.0), eps=0.0)
    np.testing.assert_allclose(y2[0], -np.arange(8.0), rtol=1e-15)
    r = np.random.default_rng(24).standard_normal((5, 16))
    g = np.random.default_rng(25).standard_normal((5, 16))
    np.testing.assert_allclose(oracle.gate_norm(7.0 * r, g, eps=0.0), oracle.gate_norm(r, g, eps=0.0),
                               rtol=1e-13)


def test_l2norm_flag():
    d = 4
    q = np.array([[[1.0, 1.0, 1.0, 1.0]], [[2.0, 0.0, 0.0, 0.0]]])
    k = np.array([[[1.0, -1.0, 1.0, -1.0]], [[0.0, 0.0, 4.0, 0.0]]])
    v = np.random.default_rng(26).standard_normal((2, 1, d))
    z = np.random.default_rng(27).standard_normal((2, 1, d))
    beta = np.array([[0.5], [0.75]])
    a = oracle.prefill(q, k, v, z, beta, np.zeros(1), qk_l2norm=True, l2_eps=0.0)
    b = oracle.prefill(q / np.linalg.norm(q, axis=-1, keepdims=True),
                       k / np.linalg.norm(k, axis=-1, keepdims=True), v, z, beta, np.zeros(1),
                       qk_l2norm=False)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------------------
# 13. Prefix-cache snapshots (Sec. 13.1): the state after every interval of a
#     sequence is the final state of a prefill of that prefix alone, and a
#     prefill resumed from it reproduces the rest of the sequence
# --------------------------------------------------------------------------

def test_snapshots_are_prefix_states():
    q, k, v, z, beta, A = _rand(407, 2, 8, seed=31)
    cu = np.array([0, 0, 130, 150, 343, 407], dtype=np.int32)   # lengths 0, 130, 20, 193, 64
    S0 = np.random.default_rng(32).standard_normal((5, 2, 8, 8))
    o, S_T, _, snaps = oracle.prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=S0, snap_interval=64)
    assert snaps.shape == (2 + 0 + 3 + 1, 2, 8, 8)
    row = 0
    for n in range(5):
        s, e = int(cu[n]), int(cu[n + 1])
        for j in range(1, (e - s) // 64 + 1):
            b = s + 64 * j
            _, Sp, _ = oracle.prefill(q[s:b], k[s:b], v[s:b], z[s:b], beta[s:b], A, S0=S0[n:n + 1])
            assert np.array_equal(snaps[row], Sp[0]), (n, j)
            o_rest, S_rest, _ = oracle.prefill(q[b:e], k[b:e], v[b:e], z[b:e], beta[b:e], A,
                                               S0=snaps[row:row + 1])
            assert np.array_equal(o_rest, o[b:e]) and np.array_equal(S_rest[0], S_T[n])
            row += 1
    assert row == snaps.shape[0]
    # the sequence of length 64 ends on a boundary: its one snapshot is its final state
    assert np.array_equal(snaps[-1], S_T[4])
    # snapshots leave the other outputs unchanged
    o2, S2, _ = oracle.prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=S0)
    assert np.array_equal(o, o2) and np.array_equal(S_T, S2)


# --------------------------------------------------------------------------
# 14. Kimi Linear's gate (Sec. 2.2, the mapping K3 replaces):
#     g = -exp(A_h) Softplus(z), unbounded below
# --------------------------------------------------------------------------

def test_softplus_gate_against_logaddexp():
    z = np.array([-60.0, -30.0, -5.0, -1e-3, 0.0, 1e-3, 0.7, 5.0, 30.0, 60.0])
    for A in (-1.0, 0.0, 0.5, 2.0):
        g = oracle.log_decay(z, A, gate="softplus")
        ref = -np.exp(A) * np.logaddexp(0.0, z)           # Softplus(z) = log(1 + e^z)
        assert np.allclose(g, ref, rtol=1e-14, atol=0.0)
        assert np.all(g < 0.0)
        assert math.isclose(g[4], -math.exp(A) * math.log(2.0), rel_tol=1e-15)
        assert math.isclose(g[-1], -math.exp(A) * 60.0, rel_tol=1e-15)   # ~ -e^A z for large z


def test_softplus_chunked_equals_recurrence():
    q, k, v, z, beta, A = _rand(150, 2, 16, seed=41, z_std=1.0)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, gate="softplus", qk_l2norm=False)
    for h in range(2):
        g = oracle.log_decay(z[:, h], A[h], gate="softplus")
        for sub in (None, 16):
            oc, Sc, _ = chunked.chunked_prefill(q[:, h], k[:, h], v[:, h], g, beta[:, h], np.zeros((16, 16)),
                                                sub=sub)
            assert np.allclose(oc, o[:, h], rtol=0, atol=1e-10 * np.abs(o[:, h]).max())
            assert np.allclose(Sc, S_T[0, h], rtol=0, atol=1e-10 * np.abs(S_T[0, h]).max())
    # the bounded gate gives a different operator on the same inputs
    o_b, _, _ = oracle.prefill(q, k, v, z, beta, A, qk_l2norm=False)
    assert not np.allclose(o_b, o)


def test_softplus_gate_breaks_the_subchunk_bound():
    """With the unbounded gate a single 16-token sub-chunk can hold a cumulative
    log decay beyond -88.7, so the factored diagonal Gram needs e^(G_a - G_j)
    above the bf16 / fp32 maximum while the exact per-pair factors stay <= 1
    and the recurrence stays finite (the page's reason for K3's bound)."""
    rng = np.random.default_rng(42)
    T, d = 64, 16
    q = _unit(rng.standard_normal((T, 1, d)))
    k = _unit(rng.standard_normal((T, 1, d)))
    v = rng.standard_normal((T, 1, d))
    z = 8.0 + rng.standard_normal((T, 1, d))             # Softplus(z) ~ 8 per step
    beta = np.full((T, 1), 0.5)
    A = np.zeros(1)
    g = oracle.log_decay(z[:, 0], A[0], gate="softplus")
    span = -np.cumsum(g[:16], axis=0)[-1]                   # decay over one sub-chunk
    assert span.max() > 88.8                                # e^span > bf16 / fp32 max
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, gate="softplus")
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(S_T))
    _, _, fmax = chunked.chunked_prefill(q[:, 0], k[:, 0], v[:, 0], g, beta[:, 0], np.zeros((d, d)), sub=16)
    assert fmax > float(np.finfo(np.float32).max)
    gb = oracle.log_decay(z[:, 0], A[0])                    # the bounded gate on the same z
    _, _, fmax_b = chunked.chunked_prefill(q[:, 0], k[:, 0], v[:, 0], gb, beta[:, 0], np.zeros((d, d)), sub=16)
    assert fmax_b < math.exp(80.0)


# --------------------------------------------------------------------------
# 15. ShortConv + Swish prologue (Sec. 2.1; Swish of Sec. 5): causal depthwise
#     conv with a conv state, pinned to library routines and invariants
# --------------------------------------------------------------------------

def test_short_conv_equals_numpy_convolve_and_expit():
    from scipy.special import expit
    from oracle import prologue
    rng = np.random.default_rng(51)
    T, C, W = 37, 6, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    y, st = prologue.short_conv(x, w, activation=False)
    for c in range(C):   # causal FIR with zero history: full convolution, first T outputs
        np.testing.assert_allclose(y[:, c], np.convolve(x[:, c], w[c, ::-1])[:T], rtol=0, atol=1e-12)
    assert np.array_equal(st[0], x[T - (W - 1):])            # state = the last W-1 inputs
    b = rng.standard_normal(C)
    ys, _ = prologue.short_conv(x, w, b)
    np.testing.assert_allclose(ys, (y + b) * expit(y + b), rtol=1e-14, atol=1e-14)
    z = np.linspace(-40, 40, 81)
    np.testing.assert_allclose(prologue.swish(z), z * expit(z), rtol=1e-14, atol=1e-300)


def test_short_conv_width_one_is_pointwise():
    from oracle import prologue
    rng = np.random.default_rng(52)
    x = rng.standard_normal((10, 5))
    w = rng.standard_normal((5, 1))
    b = rng.standard_normal(5)
    y, st = prologue.short_conv(x, w, b)
    pre = x * w[:, 0] + b
    np.testing.assert_allclose(y, pre / (1 + np.exp(-pre)), rtol=1e-14)
    assert st.shape == (1, 0, 5)


def test_short_conv_state_continuity_varlen_and_decode():
    from oracle import prologue
    rng = np.random.default_rng(53)
    T, C, W = 50, 7, 4
    x = rng.standard_normal((T, C))
    w = rng.standard_normal((C, W))
    b = rng.standard_normal(C)
    s0 = rng.standard_normal((1, W - 1, C))
    y, st = prologue.short_conv(x, w, b, state=s0)
    for a in (1, 2, 3, 17):                                   # splits shorter and longer than W-1
        y1, s1 = prologue.short_conv(x[:a], w, b, state=s0)
        y2, s2 = prologue.short_conv(x[a:], w, b, state=s1)
        assert np.array_equal(np.concatenate([y1, y2]), y) and np.array_equal(s2, st)
    # packed sequences equal separate calls
    cu = np.array([0, 0, 2, 20, 50])
    S0 = rng.standard_normal((4, W - 1, C))
    yp, sp = prologue.short_conv(x, w, b, cu_seqlens=cu, state=S0)
    for n in range(4):
        yn, sn = prologue.short_conv(x[cu[n]:cu[n + 1]], w, b, state=S0[n:n + 1])
        assert np.array_equal(yp[cu[n]:cu[n + 1]], yn) and np.array_equal(sp[n], sn[0])
    assert np.array_equal(sp[0], S0[0])                        # an empty sequence keeps its state
    # decode steps continue a prefill
    yd, sd = prologue.short_conv(x[:30], w, b, state=s0)
    for t in range(30, T):
        yt, sd = prologue.short_conv_step(x[t:t + 1], w, b, state=sd)
        assert np.array_equal(yt[0], y[t])
    assert np.array_equal(sd, st)


# --------------------------------------------------------------------------
# Mutation check: plant slips in a copy of the C oracle; the pins must notice
# --------------------------------------------------------------------------

MUTATIONS = {
    "dropped_decay": ("S[(size_t)i * dv + j] *= a;", "(void)a;"),
    "sign_of_delta": ("u[j] = bt * (vt[j] - u[j]);", "u[j] = bt * (vt[j] + u[j]);"),
    "transposed_readout": ("ot[j] += S[(size_t)i * dv + j] * qn[i];", "ot[j] += S[(size_t)j * dv + i] * qn[i];"),
    "gate_sign": ("return g_min * sigmoid(exp(A_h) * z);", "return g_min * sigmoid(-exp(A_h) * z);"),
    "snapshot_one_token_early": ("(t + 1 - cu_seqlens[n]) % snap_interval == 0",
                                 "(t + 2 - cu_seqlens[n]) % snap_interval == 0"),
    "snapshot_rows_restart": ("snap_row += (cu_seqlens[m + 1] - cu_seqlens[m]) / snap_interval;",
                              "snap_row += 0;"),
    "softplus_gate_sign": ("return -exp(A_h) * softplus(z);", "return exp(A_h) * softplus(z);"),
    "softplus_prefill_scale": ("-eA * softplus(zt[i])", "-softplus(zt[i])"),
}


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name, tmp_path):
    import ctypes
    src = open(os.path.join(os.path.dirname(oracle.__file__), "kda_oracle.c")).read()
    old, new = MUTATIONS[name]
    assert old in src
    path = tmp_path / "mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "libmut.so"
    subprocess.run(["gcc", "-O2", "-shared", "-fPIC", str(path), "-o", str(so), "-lm"], check=True)
    saved = oracle._lib
    try:
        oracle._lib = None
        lib = ctypes.CDLL(str(so))
        oracle._load()  # configure argtypes on the real library, then copy onto the mutant
        for fn in ("kda_oracle_prefill", "kda_oracle_log_decay", "kda_oracle_log_decay_softplus",
                   "kda_oracle_gate_norm"):
            getattr(lib, fn).argtypes = getattr(oracle._lib, fn).argtypes
            getattr(lib, fn).restype = getattr(oracle._lib, fn).restype
        oracle._lib = lib
        failed = False
        for pin in (lambda: test_brute_force_rational(4, 4), test_delta_invariant,
                    test_gate_closed_forms, lambda: test_chunked_equals_recurrence(150, 64, 16),
                    test_snapshots_are_prefix_states, test_softplus_gate_against_logaddexp,
                    test_softplus_chunked_equals_recurrence):
            try:
                pin()
            except AssertionError:
                failed = True
        assert failed, f"mutation {name} was not caught by the pins"
    finally:
        oracle._lib = saved
