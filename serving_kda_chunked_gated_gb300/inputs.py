"""Seeded synthetic inputs for the KDA operator workloads.

This module is shared by the tests, the benchmark and the CPU oracle's
callers.  It holds random draws, dtype packing and shape bookkeeping only:
none of the operator's arithmetic (no gate, no recurrence, no norm of an
output) lives here.  Inputs that the workloads specify as L2-normalised
(q and k) are normalised here as part of input preparation, exactly as the
workload definitions state, before they are rounded to bf16.

Every tensor of every head is drawn from its own PCG64 stream keyed by
(seed, tensor name, head), so a subset of heads of a full-size workload can
be regenerated on its own (the oracle only ever sees a few heads of the
large workloads).

Layouts (row-major, last index fastest):
  q, k        [tokens, H, dk]      bf16 bits (uint16) or float32
  v           [tokens, H, dv]      same dtype as q
  z           [tokens, H, dk]      float32 decay logits
  beta        [tokens, H]          float32, in (0, 1)
  A           [H]                  float32 per-head log scale
  S0          [N, H, dk, dv]       float32 or None (zero initial state)
  g_in        [tokens, H, dv]      bf16 bits, output-gate pre-activation
  cu_seqlens  [N + 1]              int32 token offsets of packed sequences
"""
from __future__ import annotations

import dataclasses
import zlib

import numpy as np

__all__ = [
    "Workload", "WORKLOADS", "workload", "bf16_bits", "bf16_to_f32",
    "make_prefill", "make_decode", "varlen_lengths",
]


# --------------------------------------------------------------------------
# bf16 packing (round to nearest, ties to even), data preparation only
# --------------------------------------------------------------------------

def bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round-to-nearest-even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exactly equal float32 values."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# --------------------------------------------------------------------------
# Workload definitions
# --------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" or "decode"
    H: int
    dk: int
    dv: int
    dtype: str                # "bf16" or "f32" for q, k, v (and o)
    T: int = 0                # tokens per sequence for dense prefill
    B: int = 1                # dense batch
    varlen: tuple | None = None   # (num_seqs, lo, hi) for packed varlen
    z_std: float = 1.0
    A_std: float = 0.0        # 0 -> A = 0
    S0_std: float = 0.0       # 0 -> S0 = None (zero state)
    gate: bool = False        # produce g_in for the fused output gate
    seed: int = 0


WORKLOADS = {
    # Tiny fp32 recurrence check: one head, d = 32, 64 tokens.
    "tiny": Workload("tiny", "prefill", H=1, dk=32, dv=32, dtype="f32", T=64,
                     z_std=1.0, A_std=0.0, seed=1000),
    # Single-sequence bf16 prefill, 8192 tokens, 32 heads of 128.
    "prefill_8k": Workload("prefill_8k", "prefill", H=32, dk=128, dv=128, dtype="bf16",
                           T=8192, z_std=2.0, A_std=0.5, seed=1001),
    # Long-context prefill resumed from a prefix state, with the fused gate.
    "prefill_128k": Workload("prefill_128k", "prefill", H=32, dk=128, dv=128, dtype="bf16",
                             T=131072, z_std=2.0, A_std=0.5, S0_std=0.02, gate=True,
                             seed=1002),
    # Packed variable-length prefill: 16 sequences of 512..16384 tokens.
    "varlen_16": Workload("varlen_16", "prefill", H=32, dk=128, dv=128, dtype="bf16",
                          varlen=(16, 512, 16384), z_std=2.0, A_std=0.5, seed=1003),
    # Batched single-token decode: 256 sequences, states [256, 32, 128, 128].
    "decode_256": Workload("decode_256", "decode", H=32, dk=128, dv=128, dtype="bf16",
                           B=256, z_std=2.0, A_std=0.0, S0_std=0.02, gate=True, seed=1004),
}


def workload(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (reduced sizes for tests)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


# --------------------------------------------------------------------------
# Random streams
# --------------------------------------------------------------------------

def _rng(seed: int, tensor: str, head: int) -> np.random.Generator:
    key = zlib.crc32(f"{tensor}/{head}".encode())
    return np.random.Generator(np.random.PCG64([seed, key]))


def _unit_rows(x: np.ndarray) -> np.ndarray:
    # input preparation: the workloads specify per-token L2-normalised q, k
    n = np.sqrt(np.sum(x.astype(np.float64) ** 2, axis=-1, keepdims=True))
    return (x / n).astype(np.float32)


def varlen_lengths(num_seqs: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Sequence lengths drawn uniformly from [lo, hi] (inclusive), seeded."""
    r = np.random.Generator(np.random.PCG64([seed, 0x5EC1E5]))
    return r.integers(lo, hi + 1, size=num_seqs).astype(np.int64)


def _pack(x: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits(x) if dtype == "bf16" else x.astype(np.float32)


def make_prefill(w: Workload, heads=None) -> dict:
    """Generate a prefill workload.

    heads: None for all heads, or an iterable of head indices; the result then
    holds only those heads (H' = len(heads)), with exactly the values those
    heads have in the full workload.
    """
    heads = list(range(w.H)) if heads is None else list(heads)
    if w.varlen is not None:
        n, lo, hi = w.varlen
        lens = varlen_lengths(n, lo, hi, w.seed)
    else:
        lens = np.full(w.B, w.T, dtype=np.int64)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    tok = int(cu[-1])
    Hs = len(heads)
    out = {
        "cu_seqlens": cu, "num_seqs": len(lens), "tokens": tok, "H": Hs,
        "dk": w.dk, "dv": w.dv, "dtype": w.dtype, "heads": heads,
    }
    qdt = np.uint16 if w.dtype == "bf16" else np.float32
    q = np.empty((tok, Hs, w.dk), qdt)
    k = np.empty((tok, Hs, w.dk), qdt)
    v = np.empty((tok, Hs, w.dv), qdt)
    z = np.empty((tok, Hs, w.dk), np.float32)
    beta = np.empty((tok, Hs), np.float32)
    A = np.empty((Hs,), np.float32)
    g_in = np.empty((tok, Hs, w.dv), np.uint16) if w.gate else None
    S0 = np.empty((len(lens), Hs, w.dk, w.dv), np.float32) if w.S0_std > 0 else None
    for j, h in enumerate(heads):
        q[:, j] = _pack(_unit_rows(_rng(w.seed, "q", h).standard_normal((tok, w.dk), np.float32)), w.dtype)
        k[:, j] = _pack(_unit_rows(_rng(w.seed, "k", h).standard_normal((tok, w.dk), np.float32)), w.dtype)
        v[:, j] = _pack(_rng(w.seed, "v", h).standard_normal((tok, w.dv), np.float32), w.dtype)
        z[:, j] = w.z_std * _rng(w.seed, "z", h).standard_normal((tok, w.dk), np.float32)
        b = _rng(w.seed, "beta", h).standard_normal(tok).astype(np.float64)
        beta[:, j] = (1.0 / (1.0 + np.exp(-b))).astype(np.float32)
        A[j] = np.float32(w.A_std * _rng(w.seed, "A", h).standard_normal()) if w.A_std > 0 else 0.0
        if g_in is not None:
            g_in[:, j] = bf16_bits(_rng(w.seed, "g_in", h).standard_normal((tok, w.dv), np.float32))
        if S0 is not None:
            S0[:, j] = w.S0_std * _rng(w.seed, "S0", h).standard_normal(
                (len(lens), w.dk, w.dv), np.float32)
    out.update(q=q, k=k, v=v, z=z, beta=beta, A=A, g_in=g_in, S0=S0)
    return out


def make_decode(w: Workload, heads=None, seqs=None) -> dict:
    """Generate a batched decode-step workload (one token per sequence).

    seqs: None for all B sequences, or a list of sequence indices to keep.
    """
    d = make_prefill(dataclasses.replace(w, T=1, varlen=None), heads=heads)
    if seqs is not None:
        seqs = list(seqs)
        for key in ("q", "k", "v", "z", "beta", "g_in", "S0"):
            if d[key] is not None:
                d[key] = np.ascontiguousarray(d[key][seqs])
        d["num_seqs"] = len(seqs)
        d["tokens"] = len(seqs)
        d["cu_seqlens"] = np.arange(len(seqs) + 1, dtype=np.int32)
        d["seqs"] = seqs
    d["state"] = d.pop("S0")
    return d
