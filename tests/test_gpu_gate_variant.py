"""Kimi Linear's unbounded gate g = -exp(A_h) Softplus(z) on the GPU against the
CPU oracle ("Kimi K3: KDA, attention residuals and Stable LatentMoE", Sec. 2.2,
the mapping K3's bounded gate replaces).  Under this gate a 16-token sub-chunk
can span more than the bf16/fp32 range, so the chunk-parallel prefill forms the
diagonal Gram sub-blocks pair by pair; the strong-decay cases here make the
factored form overflow."""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, qkv_to_dev, rel, to_dev

pytestmark = pytest.mark.gpu


def _case(T, H, cu=None, z=None, seed=5):
    d = I.make_prefill(I.workload("prefill_128k", T=T, H=H))
    if cu is not None:
        d["cu_seqlens"] = np.asarray(cu, dtype=np.int32)
    n = len(d["cu_seqlens"]) - 1
    d["S0"] = (0.02 * np.random.default_rng(seed).standard_normal((n, H, 128, 128))).astype(np.float32)
    if z is not None:
        d["z"] = z.astype(np.float32)
    return d


def _dev(d, dev):
    q, k, v = qkv_to_dev(d, dev)
    return dict(q=q, k=k, v=v, z=to_dev(d["z"], dev), beta=to_dev(d["beta"], dev), A=to_dev(d["A"], dev),
                cu_seqlens=to_dev(d["cu_seqlens"], dev), S0=to_dev(d["S0"], dev),
                g_in=to_dev(d["g_in"], dev, True))


def _gpu(kda, x, **kw):
    r = kda.prefill(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], cu_seqlens=x["cu_seqlens"],
                    S0=x["S0"], g_in=x["g_in"], gate="softplus", **kw)
    torch.cuda.synchronize()
    return r


def _oracle(d):
    return oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                          cu_seqlens=d["cu_seqlens"], S0=d["S0"], g_in=f64(d, "g_in"), gate="softplus")


def _check(res, ref):
    o, S_T, y = res
    ro, rS, ry = ref
    assert np.all(np.isfinite(host(o))) and np.all(np.isfinite(host(S_T)))
    assert rel(host(o), ro) < TOL_O, rel(host(o), ro)
    assert rel(host(y), ry) < TOL_O, rel(host(y), ry)
    assert rel(host(S_T), rS) < TOL_S, rel(host(S_T), rS)


CU = [0, 0, 1, 130, 150, 343, 600]


@pytest.mark.parametrize("zcase", ["workload", "strong", "mixed"])
def test_chunk_parallel_softplus_gate(kda_lib, cuda_dev, zcase):
    import serving_kda_chunked_gated_gb300.kda as kda
    rng = np.random.default_rng(11)
    shape = (CU[-1], 2, 128)
    z = {"workload": None,
         "strong": 8.0 + rng.standard_normal(shape),          # Softplus ~ 8 per step: e^-128 per sub-chunk
         "mixed": 4.0 * rng.standard_normal(shape)}[zcase]
    d = _case(CU[-1], 2, cu=CU, z=z)
    if zcase == "strong":   # the factored diagonal Gram of a sub-chunk would overflow fp32
        g = oracle.log_decay(d["z"][:16, 0], d["A"][0], gate="softplus")
        assert (-g.sum(axis=0)).max() > 88.8
    _check(_gpu(kda, _dev(d, cuda_dev)), _oracle(d))


def test_recurrent_and_decode_softplus_gate(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = _case(300, 2, cu=[0, 120, 300], z=3.0 * np.random.default_rng(12).standard_normal((300, 2, 128)))
    x = _dev(d, cuda_dev)
    _check(_gpu(kda, x, recurrent=True), _oracle(d))
    # decode: one step per sequence from the states the oracle reached
    _, rS, _ = _oracle(d)
    state = torch.from_numpy(rS.astype(np.float32)).to(cuda_dev)
    step = _case(2, 2, cu=[0, 1, 2], z=3.0 * np.random.default_rng(13).standard_normal((2, 2, 128)), seed=14)
    sx = _dev(step, cuda_dev)
    o, y = kda.decode_step(sx["q"], sx["k"], sx["v"], sx["z"], sx["beta"], sx["A"], state, g_in=sx["g_in"],
                           gate="softplus")
    torch.cuda.synchronize()
    ro, rnew, ry = oracle.decode_step(f64(step, "q"), f64(step, "k"), f64(step, "v"), step["z"], step["beta"],
                                      step["A"], rS, g_in=f64(step, "g_in"), gate="softplus")
    assert rel(host(o), ro) < TOL_O and rel(host(y), ry) < TOL_O
    assert rel(host(state), rnew) < TOL_S


def test_single_pass_schedule_rejects_softplus_gate(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = _case(200, 2)
    x = _dev(d, cuda_dev)
    small = torch.zeros(kda.PREFILL_MIN_WORKSPACE, dtype=torch.uint8, device=cuda_dev)
    with pytest.raises(kda.KDAError, match="unsupported"):
        _gpu(kda, x, workspace=small)
    cu_host = x["cu_seqlens"].cpu()            # kept alive: the args hold its address
    args = kda.make_prefill_args(x["q"], x["k"], x["v"], x["z"], x["beta"], x["A"], x["cu_seqlens"],
                                 cu_host, torch.empty_like(x["v"]), gate="softplus")
    with pytest.raises(kda.KDAError, match="unsupported"):
        kda.prefill_noalloc_raw(args)


def test_full_prefill_8k_softplus_sampled(kda_lib, cuda_dev):
    """8192 tokens x 32 heads under the Softplus gate; two heads against the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("prefill_8k")
    d = I.make_prefill(w)
    q, k, v = qkv_to_dev(d, cuda_dev)
    o, S_T, _ = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev),
                            gate="softplus")
    torch.cuda.synchronize()
    heads = [3, 30]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, _ = oracle.prefill(f64(ds, "q"), f64(ds, "k"), f64(ds, "v"), ds["z"], ds["beta"], ds["A"],
                               gate="softplus")
    assert rel(host(o)[:, heads], ro) < TOL_O
    assert rel(host(S_T)[:, heads], rS) < TOL_S
