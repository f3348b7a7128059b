"""KDA CPU oracle -- TEST INFRASTRUCTURE ONLY.

Plain, slow FP64 implementations of the Kimi Delta Attention operator used to
check the CUDA path.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does, and this package imports nothing from the product package.

  * ``kda_oracle.c``   per-token recurrence (FP64), the decay gate and the
                       output gate; built into ``_build/libkda_oracle.so``.
  * ``chunked.py``     the chunked form of the same operator in NumPy FP64,
                       with and without 16-token sub-chunk re-referencing,
                       and the KCP segment pair / combine.

Citations refer to "Kimi K3: KDA, attention residuals and Stable LatentMoE"
(hs-black.github.io): Sec. 2.1 (recurrence and chunked form), Sec. 2.2
(bounded gate, 16-token sub-chunks, e^80 bound), Sec. 2.3 (output gate),
Sec. 10.2 (KCP).

Parity status: every function here is pinned by a ``-m "not gpu"`` test in
``tests/test_oracle_pins.py`` (brute force, closed forms, invariants and the
page's printed bound values in ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libkda_oracle.so")
_lib = None

G_MIN = -5.0
L2_EPS = 1e-6
NORM_EPS = 1e-6


def build(force: bool = False) -> str:
    """Compile the C oracle with the host gcc (OpenMP when available)."""
    src = os.path.join(_HERE, "kda_oracle.c")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(src)):
        return _LIB_PATH
    os.makedirs(_BUILD, exist_ok=True)
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-fno-fast-math", "-shared", "-fPIC", src, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        d = ctypes.POINTER(ctypes.c_double)
        lib.kda_oracle_prefill.restype = None
        lib.kda_oracle_prefill.argtypes = [
            ctypes.c_int, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, ctypes.c_int, ctypes.c_int,
            d, d, d, d, d, d, ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_double,
            d, d, d, d, d, ctypes.c_double, d, ctypes.c_int, d, ctypes.c_int]
        lib.kda_oracle_log_decay.restype = ctypes.c_double
        lib.kda_oracle_log_decay.argtypes = [ctypes.c_double] * 3
        lib.kda_oracle_log_decay_softplus.restype = ctypes.c_double
        lib.kda_oracle_log_decay_softplus.argtypes = [ctypes.c_double] * 2
        lib.kda_oracle_gate_norm.restype = None
        lib.kda_oracle_gate_norm.argtypes = [d, d, d, ctypes.c_double, d, ctypes.c_long, ctypes.c_int]
        lib.kda_oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    if x is None:
        return None
    return x.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    return int(_load().kda_oracle_num_threads())


GATES = {"bounded": 0, "softplus": 1}


def log_decay(z, A_h: float, g_min: float = G_MIN, gate: str = "bounded") -> np.ndarray:
    """Decay gate of Sec. 2.2, elementwise: K3's bounded g = g_min * Sigmoid(exp(A_h) z)
    (gate="bounded"), or Kimi Linear's g = -exp(A_h) * Softplus(z) (gate="softplus")."""
    lib = _load()
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    flat, of = z.reshape(-1), out.reshape(-1)
    for i in range(flat.size):
        if GATES[gate]:
            of[i] = lib.kda_oracle_log_decay_softplus(float(flat[i]), float(A_h))
        else:
            of[i] = lib.kda_oracle_log_decay(float(flat[i]), float(A_h), float(g_min))
    return out


def prefill(q, k, v, z, beta, A, cu_seqlens=None, S0=None, g_in=None, norm_w=None,
            g_min=G_MIN, scale=1.0, qk_l2norm=True, l2_eps=L2_EPS, norm_eps=NORM_EPS,
            want_state=True, snap_interval=0, gate="bounded"):
    """Per-token recurrence, Sec. 2.1, over packed sequences.

    q, k, z: [tok, H, dk]; v: [tok, H, dv]; beta: [tok, H]; A: [H];
    cu_seqlens: int32 [N+1] (None = one sequence); S0: [N, H, dk, dv] or None.
    Returns (o [tok,H,dv], S_T [N,H,dk,dv] or None, y [tok,H,dv] or None), FP64,
    and, when snap_interval > 0, the prefix-cache snapshots [rows, H, dk, dv]:
    the state of each sequence after every snap_interval of its tokens, the
    sequences' rows in order (Sec. 13.1 prefix cache).  gate: "bounded" (K3) or
    "softplus" (Kimi Linear), see log_decay.
    """
    lib = _load()
    q, k, v, z, beta, A = map(_f64, (q, k, v, z, beta, A))
    tok, H, dk = q.shape
    dv = v.shape[2]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, tok], dtype=np.int32)
    cu = np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    N = cu.size - 1
    S0 = _f64(S0)
    g_in = _f64(g_in)
    norm_w = _f64(norm_w)
    o = np.zeros((tok, H, dv))
    S_T = np.zeros((N, H, dk, dv)) if want_state else None
    y = np.zeros((tok, H, dv)) if g_in is not None else None
    S_snap = None
    if snap_interval:
        rows = int(sum((int(cu[i + 1]) - int(cu[i])) // snap_interval for i in range(N)))
        S_snap = np.zeros((rows, H, dk, dv))
    lib.kda_oracle_prefill(
        N, cu.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), H, dk, dv,
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A),
        float(g_min), float(scale), int(bool(qk_l2norm)), float(l2_eps),
        _ptr(S0), _ptr(o), _ptr(S_T), _ptr(g_in), _ptr(norm_w), float(norm_eps), _ptr(y),
        int(snap_interval), _ptr(S_snap) if S_snap is not None and S_snap.size else None, GATES[gate])
    if snap_interval:
        return o, S_T, y, S_snap
    return o, S_T, y


def decode_step(q, k, v, z, beta, A, state, slots=None, g_in=None, norm_w=None,
                g_min=G_MIN, scale=1.0, qk_l2norm=True, l2_eps=L2_EPS, norm_eps=NORM_EPS,
                gate="bounded"):
    """One recurrent step per sequence (Sec. 2.1 with one token each).

    q, k, z: [N, H, dk]; v: [N, H, dv]; state: [S, H, dk, dv] (not modified);
    slots: int [N] rows of ``state`` (None = identity).
    Returns (o [N,H,dv], new_state [S,H,dk,dv] (a copy), y or None).
    """
    N = q.shape[0]
    state = np.asarray(state, dtype=np.float64)
    slots = np.arange(N) if slots is None else np.asarray(slots, dtype=np.int64)
    cu = np.arange(N + 1, dtype=np.int32)
    o, S_T, y = prefill(q, k, v, z, beta, A, cu_seqlens=cu, S0=state[slots], g_in=g_in,
                        norm_w=norm_w, g_min=g_min, scale=scale, qk_l2norm=qk_l2norm,
                        l2_eps=l2_eps, norm_eps=norm_eps, gate=gate)
    new_state = state.copy()
    new_state[slots] = S_T
    return o, new_state, y


def gate_norm(o, g_in, norm_w=None, eps=NORM_EPS):
    """Output gate of Sec. 2.3: y = Sigmoid(g_in) * RMSNorm(o) (per row of dv)."""
    lib = _load()
    o, g_in, norm_w = _f64(o), _f64(g_in), _f64(norm_w)
    dv = o.shape[-1]
    y = np.zeros_like(o)
    lib.kda_oracle_gate_norm(_ptr(o), _ptr(g_in), _ptr(norm_w), float(eps), _ptr(y),
                             o.size // dv, dv)
    return y
