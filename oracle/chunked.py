"""Chunked form of the KDA operator in NumPy FP64 -- TEST INFRASTRUCTURE ONLY.

Follows "Kimi K3: KDA, attention residuals and Stable LatentMoE"
(hs-black.github.io), Sec. 2.1, where the in-chunk output is

    O = (Gamma (.) Q) S + Tril[(Q (.) Gamma)(K / Gamma)^T] (U - W S),

Gamma being the cumulative product of the retentions alpha inside the chunk.
The page leaves U and W to Kimi Linear; they follow from unrolling the
recurrence inside one chunk (entry state S, rows r = 1..C, gamma_r the
inclusive cumulative retention):

    u'_r = beta_r (v_r - Sbar_r^T k_r),   Sbar_r = Diag(alpha_r) S_{r-1}
    Sbar_r = Diag(gamma_r) S + sum_{i<r} Diag(gamma_r / gamma_i) k_i u'_i^T

so (I + A) U' = Diag(beta) V - Diag(beta)(Gamma (.) K) S with
A = StrictTril(Diag(beta)(Gamma (.) K)(K / Gamma)^T); with T = (I + A)^{-1},
U = T Diag(beta) V, W = T Diag(beta)(Gamma (.) K) and U' = U - W S.  The
chunk's exit state is Diag(gamma_C) S + (K (.) gamma_C / Gamma)^T U'.

Sec. 2.2 evaluates the Gamma-ratios per 16-token sub-chunk: an entry
(i, j), i >= j, with i in sub-chunk a and j in sub-chunk b <= a, is formed as
[q_i exp(G_i - G_a)] . [k_j exp(G_a - G_j)], G_a being the cumulative log
decay at the start of sub-chunk a.  Off the diagonal both factors are <= 1;
on the diagonal the key factor is < exp(-g_min * 16) = e^80.  ``chunk_forward``
with ``sub=16`` evaluates the Gram matrices that way and reports the largest
factor it formed.

Sec. 10.2 (KCP): a segment's effect on the state is the pair (M, S~) with
S_exit = M S_entry + S~, M = M_T ... M_1, M_t = (I - beta_t k_t k_t^T)
Diag(alpha_t); pairs combine as (M2, S2) o (M1, S1) = (M2 M1, S2 + M2 S1).

Inputs here are already gated and normalised: g [T, dk] log-retentions,
q, k [T, dk], v [T, dv], beta [T], S0 [dk, dv].
"""
from __future__ import annotations

import numpy as np
from scipy.linalg import solve_triangular


def _gram_full(Qs, Ks, G):
    """Tril-able (Qs (.) Gamma)(Ks / Gamma)^T with chunk-level Gamma = exp(G)."""
    Gam = np.exp(G)
    return (Qs * Gam) @ (Ks / Gam).T, float(np.max(1.0 / Gam))


def _gram_sub(Qs, Ks, G, sub):
    """Same product, 16-token sub-chunk re-referencing (Sec. 2.2)."""
    C = Qs.shape[0]
    out = np.zeros((C, C))
    max_factor = 0.0
    nsub = (C + sub - 1) // sub
    for a in range(nsub):
        ra = slice(a * sub, min(C, (a + 1) * sub))
        Ga = G[a * sub - 1] if a > 0 else np.zeros(G.shape[1])   # log decay at start of a
        qa = Qs[ra] * np.exp(G[ra] - Ga)
        for b in range(a + 1):
            rb = slice(b * sub, min(C, (b + 1) * sub))
            fk = np.exp(Ga - G[rb])
            max_factor = max(max_factor, float(np.max(fk)))
            out[ra, rb] = qa @ (Ks[rb] * fk).T
    return out, max_factor


def chunk_forward(q, k, v, g, beta, S, sub=None):
    """One chunk: returns (O [C,dv], S_exit [dk,dv], largest Gram factor)."""
    C = q.shape[0]
    G = np.cumsum(g, axis=0)                       # inclusive, chunk-relative
    Gam = np.exp(G)
    gram = _gram_full if sub is None else (lambda a, b, c: _gram_sub(a, b, c, sub))
    Akk, f1 = gram(k, k, G)
    Akk = np.tril(beta[:, None] * Akk, -1)
    Aqk, f2 = gram(q, k, G)
    Aqk = np.tril(Aqk)
    I = np.eye(C)
    Tinv = solve_triangular(I + Akk, I, lower=True, unit_diagonal=True)
    U = Tinv @ (beta[:, None] * v)
    W = Tinv @ (beta[:, None] * (Gam * k))
    Vp = U - W @ S
    O = (q * Gam) @ S + Aqk @ Vp
    gC = Gam[-1]
    S_exit = gC[:, None] * S + (k * (gC[None, :] / Gam)).T @ Vp
    return O, S_exit, max(f1, f2)


def chunked_prefill(q, k, v, g, beta, S0, C=64, sub=None):
    """Whole sequence in chunks of C (last one partial). Returns (O, S_T, max factor)."""
    T = q.shape[0]
    S = np.array(S0, dtype=np.float64, copy=True)
    O = np.zeros((T, v.shape[1]))
    fmax = 0.0
    for s in range(0, T, C):
        e = min(T, s + C)
        O[s:e], S, f = chunk_forward(q[s:e], k[s:e], v[s:e], g[s:e], beta[s:e], S, sub)
        fmax = max(fmax, f)
    return O, S, fmax


def kcp_pair(k, v, g, beta):
    """(M, S~) of one segment, Sec. 10.2, by stepping the transition matrices."""
    dk, dv = k.shape[1], v.shape[1]
    M = np.eye(dk)
    St = np.zeros((dk, dv))
    for t in range(k.shape[0]):
        kt = k[t][:, None]
        Mt = (np.eye(dk) - beta[t] * kt @ kt.T) @ np.diag(np.exp(g[t]))
        M = Mt @ M
        St = Mt @ St + beta[t] * kt @ v[t][None, :]
    return M, St


def kcp_combine(p2, p1):
    """(M2, S2) o (M1, S1) = (M2 M1, S2 + M2 S1), Sec. 10.2."""
    M2, S2 = p2
    M1, S1 = p1
    return M2 @ M1, S2 + M2 @ S1
