"""ShortConv + Swish prologue in NumPy FP64 -- TEST INFRASTRUCTURE ONLY.

"Kimi K3: KDA, attention residuals and Stable LatentMoE" (hs-black.github.io),
Sec. 2.1: q and k pass through ShortConv, Swish and L2Norm before the
recurrence, v through ShortConv and Swish; Sec. 5 defines
Swish(z) = z * Sigmoid(z).  "Kimi-K3 深度技术分析" (liuhc.cn), the prefill-decode
section: the convolution runs along the sequence in prefill, and decode keeps a
sliding-window state of it.

Readings (the pages give no more): ShortConv is a causal depthwise 1-D
convolution of width W over each sequence's tokens, one filter per channel,
optional per-channel bias:

    pre[t, c] = sum_{i=0}^{W-1} w[c, i] * x[t - (W-1) + i, c] + b[c],
    y[t, c]   = Swish(pre[t, c])           (or pre[t, c] without activation),

where positions before a sequence's first token read that sequence's conv
state, the W-1 inputs that preceded it (oldest first), or zeros.  After the
sequence the state is the last W-1 entries of [state, x_0, ..., x_{len-1}].
"""
from __future__ import annotations

import numpy as np


def swish(z):
    """Swish(z) = z * Sigmoid(z), Sec. 5 of the KDA page."""
    z = np.asarray(z, dtype=np.float64)
    return z / (1.0 + np.exp(-z))


def short_conv(x, w, b=None, cu_seqlens=None, state=None, activation=True):
    """Causal depthwise conv over packed sequences, then Swish.

    x: [T, C]; w: [C, W]; b: [C] or None; cu_seqlens: [N+1] (None = one sequence);
    state: [N, W-1, C] or None (zeros).  Returns (y [T, C], new_state [N, W-1, C]).
    """
    x = np.asarray(x, dtype=np.float64)
    w = np.asarray(w, dtype=np.float64)
    T, C = x.shape
    W = w.shape[1]
    cu = np.array([0, T]) if cu_seqlens is None else np.asarray(cu_seqlens, dtype=np.int64)
    N = len(cu) - 1
    st = np.zeros((N, W - 1, C)) if state is None else np.asarray(state, dtype=np.float64)
    y = np.zeros((T, C))
    new_state = np.zeros((N, W - 1, C))
    for n in range(N):
        s, e = int(cu[n]), int(cu[n + 1])
        stream = np.concatenate([st[n], x[s:e]], axis=0)      # [W-1 + len, C]
        for t in range(e - s):
            window = stream[t:t + W]                          # x[t-(W-1)] .. x[t]
            pre = np.sum(window * w.T, axis=0)
            if b is not None:
                pre = pre + b
            y[s + t] = swish(pre) if activation else pre
        new_state[n] = stream[len(stream) - (W - 1):] if W > 1 else np.zeros((0, C))
    return y, new_state


def short_conv_step(x, w, b=None, state=None, slots=None, activation=True):
    """One decode step: x [N, C] (one token per sequence), state [S, W-1, C]
    (not modified; rows `slots`, None = identity).  Returns (y [N, C], new_state)."""
    x = np.asarray(x, dtype=np.float64)
    N = x.shape[0]
    state = np.asarray(state, dtype=np.float64)
    slots = np.arange(N) if slots is None else np.asarray(slots)
    y, ns = short_conv(x, w, b, cu_seqlens=np.arange(N + 1), state=state[slots], activation=activation)
    new_state = state.copy()
    new_state[slots] = ns
    return y, new_state
