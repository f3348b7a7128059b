"""Randomised properties of the FP64 oracle (hypothesis; skipped where it is not
installed): the chunked form of Sec. 2.1 equals the recurrence for any length,
width, chunk and sub-chunk size and decay strength; the operator is jointly
linear in (v, S0); packing sequences together and splitting one at any point
change nothing (bit for bit in the C recurrence)."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402
from oracle import chunked  # noqa: E402

SETTINGS = settings(max_examples=30, deadline=None)


def _inputs(seed, T, H, d, z_std):
    r = np.random.default_rng(seed)
    q = r.standard_normal((T, H, d))
    k = r.standard_normal((T, H, d))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = r.standard_normal((T, H, d))
    z = z_std * r.standard_normal((T, H, d))
    beta = 1 / (1 + np.exp(-r.standard_normal((T, H))))
    A = 0.5 * r.standard_normal(H)
    S0 = 0.3 * r.standard_normal((1, H, d, d))
    return q, k, v, z, beta, A, S0


@SETTINGS
@given(seed=st.integers(0, 2**31 - 1), T=st.integers(1, 100), d=st.integers(2, 8),
       C=st.sampled_from([8, 16, 32, 64]), sub=st.sampled_from([None, 4, 8, 16]),
       z_std=st.sampled_from([0.5, 2.0, 4.0]))
def test_chunked_equals_recurrence_randomised(seed, T, d, C, sub, z_std):
    if sub is not None and sub > C:
        sub = None
    q, k, v, z, beta, A, S0 = _inputs(seed, T, 1, d, z_std)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    g = oracle.log_decay(z[:, 0], A[0])
    O, S, _ = chunked.chunked_prefill(q[:, 0], k[:, 0], v[:, 0], g, beta[:, 0], S0[0, 0], C=C, sub=sub)
    np.testing.assert_allclose(O, o[:, 0], rtol=0, atol=1e-10 * max(1.0, np.abs(o).max()))
    np.testing.assert_allclose(S, S_T[0, 0], rtol=0, atol=1e-10 * max(1.0, np.abs(S_T).max()))


@SETTINGS
@given(seed=st.integers(0, 2**31 - 1), T=st.integers(1, 60), H=st.integers(1, 3), d=st.integers(2, 8))
def test_linear_in_values_and_initial_state(seed, T, H, d):
    """o and S_T are linear in (v, S0) jointly: f(v, S0) = f(v, 0) + f(0, S0)."""
    q, k, v, z, beta, A, S0 = _inputs(seed, T, H, d, 2.0)
    o, S, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    o1, S1, _ = oracle.prefill(q, k, v, z, beta, A, S0=None, qk_l2norm=False)
    o2, S2, _ = oracle.prefill(q, k, np.zeros_like(v), z, beta, A, S0=S0, qk_l2norm=False)
    scale = max(1.0, np.abs(o).max(), np.abs(S).max())
    np.testing.assert_allclose(o, o1 + o2, rtol=0, atol=1e-12 * scale)
    np.testing.assert_allclose(S, S1 + S2, rtol=0, atol=1e-12 * scale)


@SETTINGS
@given(seed=st.integers(0, 2**31 - 1), lens=st.lists(st.integers(0, 40), min_size=1, max_size=4),
       d=st.integers(2, 6))
def test_packing_changes_nothing(seed, lens, d):
    """Packed sequences (empty ones included) give each sequence's own result, bit for bit."""
    T = sum(lens)
    H = 2
    q, k, v, z, beta, A, _ = _inputs(seed, T, H, d, 2.0)
    S0 = 0.3 * np.random.default_rng(seed + 1).standard_normal((len(lens), H, d, d))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=S0, qk_l2norm=False)
    for n in range(len(lens)):
        s, e = cu[n], cu[n + 1]
        on, Sn, _ = oracle.prefill(q[s:e], k[s:e], v[s:e], z[s:e], beta[s:e], A, S0=S0[n:n + 1],
                                   qk_l2norm=False)
        assert np.array_equal(o[s:e], on) and np.array_equal(S_T[n], Sn[0])


@SETTINGS
@given(seed=st.integers(0, 2**31 - 1), T=st.integers(2, 80), cut=st.floats(0.0, 1.0), d=st.integers(2, 6))
def test_split_anywhere_and_resume(seed, T, cut, d):
    """A prefill split at any token and resumed from the state it left is the whole prefill, bit for bit."""
    t = int(round(cut * T))
    q, k, v, z, beta, A, S0 = _inputs(seed, T, 2, d, 2.0)
    o, S_T, _ = oracle.prefill(q, k, v, z, beta, A, S0=S0, qk_l2norm=False)
    o1, S1, _ = oracle.prefill(q[:t], k[:t], v[:t], z[:t], beta[:t], A, S0=S0, qk_l2norm=False)
    o2, S2, _ = oracle.prefill(q[t:], k[t:], v[t:], z[t:], beta[t:], A, S0=S1, qk_l2norm=False)
    assert np.array_equal(np.concatenate([o1, o2]), o) and np.array_equal(S2, S_T)
