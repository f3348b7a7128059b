"""Helpers shared by the GPU parity tests (conversions and error measures).

Every comparison of a GPU result with the oracle goes through ``parity``,
which checks, on top of the global relative L2 error the operator's tolerance
is stated in (2e-3 on o and y, 1e-3 on final states):

  * no non-finite value in the GPU result;
  * a per-row bound: every row (one (token, head) output vector over d_v, or
    one row of a d_k x d_v state) has a relative L2 error below ROW_TOL, so a
    wrong tail or a wrong head cannot hide inside a large global norm.  Rows
    whose reference norm is tiny compared with the typical row of their head
    (below ROW_FLOOR times the head's root-mean-square row norm over the
    tokens) are measured against that floor instead of their own norm: the
    arithmetic error of a row scales with the head's state, not with the row's
    own output, which can be small by cancellation.  The fused output y = Sigmoid(g) (.)
    RMSNorm(o) rescales every row to about the same norm, so the relative
    error of a y row equals that of its o row; the y rows take the floor of the
    o rows they come from (their error is weighted by |o_r| / max(|o_r|, floor));
  * optionally, the global error of each packed sequence on its own;
  * for bf16 outputs, two figures printed beside the check: the error
    against the oracle rounded to bf16, and the arithmetic error estimated in
    quadrature, sqrt(rel^2 - storage^2), where storage is what rounding the
    exact result to bf16 costs by itself (about 1.7e-3).  Neither is asserted:
    the first counts whole-ulp flips of values near a rounding boundary, so it
    grows like the square root of the arithmetic error, and the second is noisy
    on small outputs.
"""
import numpy as np
import torch

from serving_kda_chunked_gated_gb300 import inputs as I

TOL_O = 2e-3      # relative L2 on o (and y), bf16 outputs
TOL_S = 1e-3      # relative L2 on final states
ROW_TOL = 2e-2    # relative L2 of any single row
ROW_FLOOR = 0.1   # rows with norms below this fraction of their head's rms row norm use the floor


def rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return float(np.linalg.norm(a - b) / nb) if nb > 0 else float(np.linalg.norm(a))


def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), as the GPU's stores do."""
    return I.bf16_to_f32(I.bf16_bits(np.asarray(x, dtype=np.float32))).astype(np.float64)


def _floored(rn):
    """rn: row norms shaped [tokens or sequences, ...groups]; the floor of each
    group (a head) is ROW_FLOOR times its rms over axis 0."""
    rms = np.sqrt(np.mean(rn * rn, axis=0, keepdims=True)) if rn.size else np.zeros_like(rn)
    den = np.maximum(rn, ROW_FLOOR * rms)
    den[den == 0] = 1.0
    return den


def row_errors(got, ref, floor_ref=None) -> np.ndarray:
    """Relative L2 error of every row (last axis), with the small-row floor;
    with floor_ref (the rows a normalised output comes from), the floor of
    floor_ref's rows applies instead."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    if g.ndim == 1:
        g, r = g[None], r[None]
    rn = np.linalg.norm(r, axis=-1)           # [axis 0, ...groups]
    err = np.linalg.norm(g - r, axis=-1)
    if floor_ref is None:
        return err / _floored(rn)
    fn = np.linalg.norm(np.asarray(floor_ref, dtype=np.float64), axis=-1)
    rn = rn.copy()
    rn[rn == 0] = 1.0
    return err / rn * (fn / _floored(fn))


def parity(name, got, ref, tol, bf16_out=False, seq_bounds=None, row_tol=ROW_TOL, floor_ref=None):
    """Assert that ``got`` (GPU) matches ``ref`` (oracle, FP64); see the module
    docstring.  seq_bounds: sequence boundaries along axis 0 (cu_seqlens for
    token-major outputs, range(N + 1) for per-sequence states); floor_ref: for
    the fused output y, the oracle's o.  Returns the measured figures and
    prints them on one line."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, f"{name}: shape {got.shape} vs {ref.shape}"
    bad = int(np.count_nonzero(~np.isfinite(got)))
    assert bad == 0, f"{name}: {bad} non-finite values"
    e = rel(got, ref)
    rows = row_errors(got, ref, floor_ref)
    r_max = float(rows.max()) if rows.size else 0.0
    out = {"rel": e, "row_max": r_max}
    where = np.unravel_index(int(np.argmax(rows)), rows.shape) if rows.size else ()
    msg = (f"{name}: rel-L2 {e:.3e} (tol {tol:.0e}), max row {r_max:.3e} at {tuple(int(i) for i in where)}"
           f" (tol {row_tol:.0e})")
    if bf16_out:
        rb = bf16_round(ref)
        out["rel_vs_bf16_ref"] = rel(got, rb)
        out["bf16_storage"] = rel(rb, ref)
        out["arith_est"] = float(np.sqrt(max(0.0, e * e - out["bf16_storage"] ** 2)))
        msg += (f", vs bf16(oracle) {out['rel_vs_bf16_ref']:.3e}, bf16 storage alone"
                f" {out['bf16_storage']:.3e}, arithmetic ~{out['arith_est']:.1e}")
    worst_seq = None
    if seq_bounds is not None:
        sb = [int(x) for x in seq_bounds]
        errs = [(rel(got[s:t], ref[s:t]), i) for i, (s, t) in enumerate(zip(sb[:-1], sb[1:])) if t > s]
        if errs:
            worst_seq = max(errs)
            out["seq_max"] = worst_seq[0]
            msg += f", worst sequence {worst_seq[1]}: {worst_seq[0]:.3e}"
    print(msg)
    assert e < tol, msg
    assert r_max <= row_tol, msg
    if worst_seq is not None:
        assert worst_seq[0] < tol, msg
    return out


def to_dev(x, dev, bf16=False):
    if x is None:
        return None
    if bf16:
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).to(dev)
    return torch.from_numpy(np.ascontiguousarray(x)).to(dev)


def qkv_to_dev(d, dev):
    bf = d["dtype"] == "bf16"
    return (to_dev(d["q"], dev, bf), to_dev(d["k"], dev, bf), to_dev(d["v"], dev, bf))


def f64(d, key):
    x = d[key]
    if x is None:
        return None
    if x.dtype == np.uint16:
        return I.bf16_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def host(t):
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
