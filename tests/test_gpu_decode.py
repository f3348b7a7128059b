"""Decode step on the GPU against the CPU oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, rel, to_dev

pytestmark = pytest.mark.gpu


def _run(kda, d, dev, slots=None, state=None, gate=True, want_o=True):
    st = to_dev(d["state"].copy(), dev) if state is None else state
    sl = to_dev(np.asarray(slots, dtype=np.int32), dev) if slots is not None else None
    o, y = kda.decode_step(to_dev(d["q"], dev, True), to_dev(d["k"], dev, True), to_dev(d["v"], dev, True),
                           to_dev(d["z"], dev), to_dev(d["beta"], dev), to_dev(d["A"], dev), st,
                           g_in=to_dev(d["g_in"], dev, True) if gate else None, slots=sl, want_o=want_o)
    torch.cuda.synchronize()
    return o, y, st


def test_decode_small_against_oracle(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_decode(I.workload("decode_256", H=4, B=16))
    o, y, st = _run(kda, d, cuda_dev)
    ro, rs, ry = oracle.decode_step(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                    d["state"], g_in=f64(d, "g_in"))
    assert rel(host(o), ro) < TOL_O
    assert rel(host(y), ry) < TOL_O
    assert rel(host(st), rs) < TOL_S
    # element-wise: the state is FP32 throughout, so every element is close
    np.testing.assert_allclose(host(st), rs, rtol=0, atol=2e-5)


def test_decode_slots_permuted_and_skipped(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_decode(I.workload("decode_256", H=2, B=6))
    pool = np.random.default_rng(0).standard_normal((10, 2, 128, 128)).astype(np.float32) * 0.02
    slots = np.array([7, 2, 9, 0, 4, 5], dtype=np.int32)
    st = to_dev(pool.copy(), cuda_dev)
    o, y, st = _run(kda, d, cuda_dev, slots=slots, state=st)
    ro, rs, ry = oracle.decode_step(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                    pool, slots=slots, g_in=f64(d, "g_in"))
    assert rel(host(st), rs) < TOL_S and rel(host(o), ro) < TOL_O and rel(host(y), ry) < TOL_O
    untouched = [1, 3, 6, 8]
    assert np.array_equal(host(st)[untouched], pool[untouched])
    # an out-of-range slot is skipped by the kernel's range check: its outputs stay untouched
    bad = slots.copy()
    bad[2] = 10
    st2 = to_dev(pool.copy(), cuda_dev)
    o2, y2, st2 = _run(kda, d, cuda_dev, slots=bad, state=st2)
    good = [0, 1, 3, 4, 5]
    np.testing.assert_allclose(host(o2)[good], host(o)[good], rtol=0, atol=0)
    assert np.array_equal(host(st2)[9], pool[9])


def test_decode_full_size_sampled(kda_lib, cuda_dev):
    """Full decode workload (256 sequences x 32 heads); the oracle checks sampled pairs."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("decode_256")
    d = I.make_decode(w)
    o, y, st = _run(kda, d, cuda_dev)
    # run twice from the same start: bit-identical (no atomics on any output path)
    o_b, y_b, st_b = _run(kda, d, cuda_dev)
    assert torch.equal(st, st_b) and torch.equal(y, y_b)
    heads = [0, 13, 31]
    seqs = [0, 77, 255]
    ds = I.make_decode(w, heads=heads, seqs=seqs)
    ro, rs, ry = oracle.decode_step(f64(ds, "q"), f64(ds, "k"), f64(ds, "v"), ds["z"], ds["beta"],
                                    ds["A"], ds["state"], g_in=f64(ds, "g_in"))
    sub = np.ix_(seqs, heads)
    assert rel(host(o)[sub], ro) < TOL_O
    assert rel(host(y)[sub], ry) < TOL_O
    assert rel(host(st)[sub], rs) < TOL_S


def test_decode_y_only(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_decode(I.workload("decode_256", H=2, B=3))
    o, y, st = _run(kda, d, cuda_dev, want_o=False)
    assert o is None
    _, _, ry = oracle.decode_step(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                  d["state"], g_in=f64(d, "g_in"))
    assert rel(host(y), ry) < TOL_O


def test_decode_normalises_raw_q_k(kda_lib, cuda_dev):
    """q and k NOT normalised (each token-head vector scaled by a factor in
    0.2..5) with qk_l2norm on: the kernel's own L2 norm of q and k matches the
    oracle's, element by element on the state."""
    import serving_kda_chunked_gated_gb300.kda as kda
    from kda_testutil import parity
    d = I.make_decode(I.workload("decode_256", H=4, B=16))
    rng = np.random.default_rng(3)
    for key in ("q", "k"):
        f = rng.uniform(0.2, 5.0, size=(16, 4, 1)).astype(np.float32)
        d[key] = I.bf16_bits(I.bf16_to_f32(d[key]) * f)
    o, y, st = _run(kda, d, cuda_dev)
    ro, rs, ry = oracle.decode_step(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                    d["state"], g_in=f64(d, "g_in"), qk_l2norm=True)
    parity("o", host(o), ro, TOL_O, bf16_out=True)
    parity("y", host(y), ry, TOL_O, bf16_out=True, floor_ref=ro)
    parity("state", host(st), rs, TOL_S)
    np.testing.assert_allclose(host(st), rs, rtol=0, atol=2e-5)
    # without the norm the same inputs give a different result: the flag is read
    st2 = to_dev(d["state"].copy(), cuda_dev)
    o2, _ = kda.decode_step(to_dev(d["q"], cuda_dev, True), to_dev(d["k"], cuda_dev, True),
                            to_dev(d["v"], cuda_dev, True), to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev),
                            to_dev(d["A"], cuda_dev), st2, qk_l2norm=False)
    torch.cuda.synchronize()
    assert rel(host(o2), ro) > 0.1
