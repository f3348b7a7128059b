"""Seeded input generator: bf16 packing, determinism, head-subset regeneration."""
import numpy as np

from serving_kda_chunked_gated_gb300 import inputs as I


def test_bf16_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e38, 1e-40], dtype=np.float32)
    b = I.bf16_bits(x)
    assert list(b[:4]) == [0x3F80, 0x3F80, 0x3F82, 0xC020]
    back = I.bf16_to_f32(b)
    assert back[0] == 1.0 and back[3] == -2.5
    r = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    err = np.abs(I.bf16_to_f32(I.bf16_bits(r)) - r) / np.abs(r)
    assert err.max() <= 2 ** -8 + 1e-9


def test_deterministic_and_head_subset():
    w = I.workload("prefill_8k", T=100, H=4)
    a = I.make_prefill(w)
    b = I.make_prefill(w)
    for key in ("q", "k", "v", "z", "beta", "A"):
        assert np.array_equal(a[key], b[key])
    s = I.make_prefill(w, heads=[3, 1])
    for key in ("q", "k", "v", "z"):
        assert np.array_equal(s[key][:, 0], a[key][:, 3]) and np.array_equal(s[key][:, 1], a[key][:, 1])
    assert np.array_equal(s["beta"][:, 0], a["beta"][:, 3])
    qn = np.linalg.norm(I.bf16_to_f32(a["q"]).astype(np.float64), axis=-1)
    assert np.allclose(qn, 1.0, atol=1e-2)
    assert np.all((a["beta"] > 0) & (a["beta"] < 1))


def test_varlen_lengths():
    w = I.workload("varlen_16")
    lens = I.varlen_lengths(*w.varlen, w.seed)
    assert lens.shape == (16,) and lens.min() >= 512 and lens.max() <= 16384
    d = I.make_prefill(I.workload("varlen_16", H=1))
    assert d["cu_seqlens"][0] == 0 and np.all(np.diff(d["cu_seqlens"]) == lens)


def test_decode_shapes():
    d = I.make_decode(I.workload("decode_256", H=2, B=5))
    assert d["q"].shape == (5, 2, 128) and d["state"].shape == (5, 2, 128, 128)
    assert d["g_in"].shape == (5, 2, 128) and np.all(d["A"] == 0)
