"""Prefix-cache state snapshots on the GPU against the CPU oracle.

A prefill with snapshots writes the FP32 state of every sequence after each
snap_interval of its tokens ("Kimi K3: KDA, attention residuals and Stable
LatentMoE", Sec. 13.1: a cached prefix is reusable only where its recurrent
state can be restored at the same boundary).  Checked here: the snapshots
equal the oracle's states at those boundaries, a prefill resumed from any of
them reproduces the rest of the sequence, and asking for snapshots changes no
other output."""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, qkv_to_dev, rel, to_dev

pytestmark = pytest.mark.gpu


def _dev_inputs(d, dev):
    q, k, v = qkv_to_dev(d, dev)
    return dict(q=q, k=k, v=v, z=to_dev(d["z"], dev), beta=to_dev(d["beta"], dev),
                A=to_dev(d["A"], dev), cu_seqlens=to_dev(d["cu_seqlens"], dev),
                S0=to_dev(d["S0"], dev) if d["S0"] is not None else None,
                g_in=to_dev(d["g_in"], dev, True) if d["g_in"] is not None else None)


def _gpu(kda, x, **kw):
    r = kda.prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                    S0=x["S0"], g_in=x["g_in"], **kw)
    torch.cuda.synchronize()
    return r


def _oracle(d, interval):
    return oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                          cu_seqlens=d["cu_seqlens"], S0=d["S0"], g_in=f64(d, "g_in"),
                          snap_interval=interval)


def _varlen(H, cu, seed=3, dtype_workload="prefill_128k"):
    d = I.make_prefill(I.workload(dtype_workload, T=int(cu[-1]), H=H))
    d["cu_seqlens"] = np.asarray(cu, dtype=np.int32)
    n = len(cu) - 1
    dk, dv = d["q"].shape[2], d["v"].shape[2]
    d["S0"] = (0.02 * np.random.default_rng(seed).standard_normal((n, H, dk, dv))).astype(np.float32)
    return d


# sequence lengths 0, 130, 20, 193, 64, 256: empty, ragged, shorter than one
# interval, ending exactly on a boundary
CU = [0, 0, 130, 150, 343, 407, 663]


@pytest.mark.parametrize("interval", [64, 128])
def test_snapshots_match_oracle_tensor_core(kda_lib, cuda_dev, interval):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = _varlen(2, CU)
    x = _dev_inputs(d, cuda_dev)
    o, S_T, y, snaps = _gpu(kda, x, snap_interval=interval)
    ro, rS, ry, rsnap = _oracle(d, interval)
    assert snaps.shape == rsnap.shape == (kda.snapshot_count(CU, interval), 2, 128, 128)
    for j in range(snaps.shape[0]):
        assert rel(host(snaps[j]), rsnap[j]) < TOL_S, f"snapshot {j}"
    assert rel(host(o), ro) < TOL_O and rel(host(y), ry) < TOL_O and rel(host(S_T), rS) < TOL_S
    # a sequence that ends on a boundary: its last snapshot is its final state, bit for bit
    assert torch.equal(snaps[-1], S_T[5])
    # snapshots change nothing else
    o2, S2, y2 = _gpu(kda, x)
    assert torch.equal(o, o2) and torch.equal(S_T, S2) and torch.equal(y, y2)


def test_snapshots_match_oracle_recurrent_paths(kda_lib, cuda_dev):
    """The per-token kernel (float32 inputs with d = 32, and bf16 forced onto
    it) emits the same rows."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d32 = I.make_prefill(I.workload("tiny", T=200))
    d32["cu_seqlens"] = np.array([0, 5, 200], dtype=np.int32)      # 5 tokens, then 195
    d32["S0"] = (0.1 * np.random.default_rng(4).standard_normal((2, 1, 32, 32))).astype(np.float32)
    for d, rec in ((d32, False), (_varlen(2, CU), True)):
        x = _dev_inputs(d, cuda_dev)
        o, S_T, y, snaps = _gpu(kda, x, snap_interval=64, recurrent=rec)
        ro, rS, ry, rsnap = _oracle(d, 64)
        assert snaps.shape == rsnap.shape and snaps.shape[0] == kda.snapshot_count(d["cu_seqlens"], 64)
        assert rel(host(snaps), rsnap) < TOL_S
        assert rel(host(o), ro) < TOL_O and rel(host(S_T), rS) < TOL_S


def test_resume_from_every_snapshot(kda_lib, cuda_dev):
    """Resuming sequence 3 (193 tokens) from each of its snapshots reproduces
    its remaining outputs and final state (the cache-hit path: prefill only the
    uncached suffix)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = _varlen(2, CU)
    x = _dev_inputs(d, cuda_dev)
    o, S_T, y, snaps = _gpu(kda, x, snap_interval=64)
    ro, rS, ry, _ = _oracle(d, 64)
    s, e = CU[3], CU[4]
    base = kda.snapshot_count(CU[:4], 64)
    for j in range(1, (e - s) // 64 + 1):
        b = s + 64 * j
        sl = slice(b, e)
        c = lambda t: t[sl].clone()
        o_r, S_r, y_r = kda.prefill(c(x["q"]), c(x["k"]), c(x["v"]), c(x["z"]), c(x["beta"]), x["A"],
                                    S0=snaps[base + j - 1:base + j].clone(), g_in=c(x["g_in"]))
        torch.cuda.synchronize()
        assert rel(host(o_r), ro[sl]) < TOL_O and rel(host(y_r), ry[sl]) < TOL_O
        assert rel(host(S_r[0]), rS[3]) < TOL_S
        assert rel(host(o_r), host(o[sl])) < TOL_O


def test_full_varlen_16_snapshots_sampled(kda_lib, cuda_dev):
    """Packed 16-sequence prefill (lengths 512..16384) with a snapshot every
    1024 tokens: two heads of every snapshot row checked against the oracle;
    the other outputs are bit-identical to a run without snapshots."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("varlen_16")
    d = I.make_prefill(w)
    x = _dev_inputs(d, cuda_dev)
    o, S_T, _, snaps = _gpu(kda, x, snap_interval=1024)
    o2, S2, _ = _gpu(kda, x)
    assert torch.equal(o, o2) and torch.equal(S_T, S2)
    cu = d["cu_seqlens"]
    assert snaps.shape[0] == kda.snapshot_count(cu, 1024) > 16
    del x, o2, S2
    heads = [0, 31]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, _, rsnap = _oracle(ds, 1024)
    assert rel(host(snaps[:, heads]), rsnap) < TOL_S
    assert rel(host(S_T[:, heads]), rS) < TOL_S
