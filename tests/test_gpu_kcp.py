"""KDA context parallelism (Sec. 10.2) on the GPU: the transition pair of a
segment from two state-only prefills, kda_kcp_apply, and the one-device KCP
driver (ranks taken in turn) against the single-pass prefill and the oracle."""
import numpy as np
import pytest
import torch

import oracle
from oracle import chunked
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, qkv_to_dev, rel, to_dev

pytestmark = pytest.mark.gpu


def _segments(d, dev, cuts):
    q, k, v = qkv_to_dev(d, dev)
    z, beta = to_dev(d["z"], dev), to_dev(d["beta"], dev)
    A = to_dev(d["A"], dev)
    segs = []
    for i in range(len(cuts) - 1):
        sl = slice(cuts[i], cuts[i + 1])
        segs.append(dict(q=q[sl].clone(), k=k[sl].clone(), v=v[sl].clone(), z=z[sl].clone(), beta=beta[sl].clone(),
                         A=A))
    return segs


def test_pair_from_state_only_prefills(kda_lib, cuda_dev):
    """M of a short, weakly decaying segment (over long segments of the workload's
    decays M underflows fp32: the pairs' M carries no memory there)."""
    from serving_kda_chunked_gated_gb300 import kcp
    d = I.make_prefill(I.workload("prefill_128k", T=100, H=2))
    d["z"] = (d["z"] - 4.0).astype(np.float32)
    seg = _segments(d, cuda_dev, [0, 100])[0]
    M, St = kcp.GpuOps().pair(seg)
    torch.cuda.synchronize()
    qn = f64(d, "q")
    kn = f64(d, "k")
    kn = kn / np.sqrt((kn * kn).sum(-1, keepdims=True) + 1e-6)   # the prefill's L2Norm of k
    X = 0.02 * np.random.default_rng(7).standard_normal((128, 128))   # a state of the workload's scale
    for h in range(2):
        g = oracle.log_decay(d["z"][:, h], d["A"][h])
        rM, rSt = chunked.kcp_pair(kn[:, h], f64(d, "v")[:, h], g, d["beta"][:, h].astype(np.float64))
        assert rel(host(St[h]), rSt) < TOL_S
        # the fold the pair exists for: S <- M S + S~
        assert rel(host(M[h]) @ X + host(St[h]), rM @ X + rSt) < TOL_S
        # M itself: relative, or, once it has decayed below 2^-14 of |S0| = |I|,
        # relative to that (the scan's fp16 record operands hold terms down to
        # 2^-24 of their own scale; one head here decays to |M| ~ 1e-27)
        err = np.linalg.norm(host(M[h]) - rM)
        assert err <= TOL_S * max(np.linalg.norm(rM), 2.0 ** -14 * np.sqrt(128)), err


@pytest.mark.parametrize("n", [128, 256, 40])
def test_kcp_apply(kda_lib, cuda_dev, n):
    import serving_kda_chunked_gated_gb300.kda as kda
    g = torch.Generator().manual_seed(n)
    H, dd = 3, 128
    M = torch.randn((H, dd, dd), generator=g) / 12
    X = torch.randn((H, dd, n), generator=g)
    add = torch.randn((H, dd, n), generator=g)
    ref = torch.matmul(M.double(), X.double()) + add.double()
    Xd = X.to(cuda_dev)
    kda.kcp_apply(M.to(cuda_dev), Xd, add.to(cuda_dev))
    torch.cuda.synchronize()
    assert rel(Xd.cpu().numpy(), ref.numpy()) < 1e-6
    X2 = X.to(cuda_dev)
    kda.kcp_apply(M.to(cuda_dev), X2)
    torch.cuda.synchronize()
    assert rel(X2.cpu().numpy(), torch.matmul(M.double(), X.double()).numpy()) < 1e-6


def test_local_kcp_matches_single_pass_and_oracle(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    from serving_kda_chunked_gated_gb300 import kcp
    T, cuts = 1000, [0, 250, 251, 700, 1000]
    d = I.make_prefill(I.workload("prefill_128k", T=T, H=2))
    segs = _segments(d, cuda_dev, cuts)
    outs = kcp.kcp_prefill_local(segs, kcp.GpuOps())
    q, k, v = qkv_to_dev(d, cuda_dev)
    o1, S1, _ = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev))
    torch.cuda.synchronize()
    o = torch.cat([x[0] for x in outs])
    assert rel(host(o), host(o1)) < TOL_O and rel(host(outs[-1][1]), host(S1[0])) < TOL_S
    ro, rS, _ = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"])
    assert rel(host(o), ro) < TOL_O and rel(host(outs[-1][1]), rS[0]) < TOL_S


def test_local_kcp_full_size_eight_segments(kda_lib, cuda_dev):
    """131072 tokens x 32 heads in eight 16384-token segments: the KCP result
    equals the single-pass prefill, and one head equals the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    from serving_kda_chunked_gated_gb300 import kcp
    w = I.workload("prefill_128k")
    d = I.make_prefill(w)
    T = d["q"].shape[0]
    cuts = list(range(0, T + 1, T // 8))
    segs = _segments(d, cuda_dev, cuts)
    outs = kcp.kcp_prefill_local(segs, kcp.GpuOps())
    o = torch.cat([x[0] for x in outs])
    S_kcp = outs[-1][1]
    del segs, outs
    q, k, v = qkv_to_dev(d, cuda_dev)
    o1, S1, _ = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev))
    torch.cuda.synchronize()
    assert rel(host(o), host(o1)) < TOL_O and rel(host(S_kcp), host(S1[0])) < TOL_S
    heads = [9]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, _ = oracle.prefill(f64(ds, "q"), f64(ds, "k"), f64(ds, "v"), ds["z"], ds["beta"], ds["A"])
    assert rel(host(o[:, heads]), ro) < TOL_O and rel(host(S_kcp[heads]), rS[0]) < TOL_S


def test_records_then_scans_equal_prefill(kda_lib, cuda_dev):
    """kda_prefill_records + kda_prefill_scan give kda_prefill's results bit for
    bit (packed ragged sequences incl. an empty one, S0, the fused gate), several
    scans over one set of records agree, and the zero-v scan equals a prefill
    with v = 0 (the KCP transition M)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    cu = [0, 1, 130, 130, 449, 700]
    H = 3
    d = I.make_prefill(I.workload("prefill_128k", T=cu[-1], H=H))
    q, k, v = qkv_to_dev(d, cuda_dev)
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    cu_d = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    S0 = torch.randn((len(cu) - 1, H, 128, 128), generator=torch.Generator().manual_seed(5)).to(cuda_dev) / 8
    g_in = torch.randn((cu[-1], H, 128), generator=torch.Generator().manual_seed(6)).to(cuda_dev).to(torch.bfloat16)
    o1, S1, y1 = kda.prefill(q, k, v, z, beta, A, cu_seqlens=cu_d, S0=S0, g_in=g_in)
    rec = kda.prefill_records(q, k, v, z, beta, A, cu_seqlens=cu_d)
    for _ in range(2):
        o2, S2, y2 = kda.prefill_scan(rec, S0=S0, g_in=g_in)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(S1, S2) and torch.equal(y1, y2)
    _, Sz, _ = kda.prefill_scan(rec, want_o=False)                       # from zero, records reused
    _, Sz1, _ = kda.prefill(q, k, v, z, beta, A, cu_seqlens=cu_d, want_o=False)
    assert torch.equal(Sz, Sz1)
    # bit for bit here: over these 700 tokens the largest |S| stays within [2^-6, 2^6]
    # of its starting scale, so the zero-v (transition) scan never moves its
    # state exponent and computes exactly what the plain scan does
    o3, S3, _ = kda.prefill_scan(rec, S0=S0, zero_v=True)
    o4, S4, _ = kda.prefill(q, k, torch.zeros_like(v), z, beta, A, cu_seqlens=cu_d, S0=S0)
    torch.cuda.synchronize()
    assert torch.equal(o3, o4) and torch.equal(S3, S4)


def test_local_kcp_without_records_fp32(kda_lib, cuda_dev):
    """fp32 inputs with d = 64 have no chunk-parallel schedule: GpuOps then takes
    three kda_prefill calls per segment (per-token recurrence); the KCP result
    still equals the single pass and the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    from serving_kda_chunked_gated_gb300 import kcp
    T, cuts = 300, [0, 100, 101, 300]
    d = I.make_prefill(I.workload("tiny", T=T, H=2, dk=64, dv=64))
    segs = _segments(d, cuda_dev, cuts)
    ops = kcp.GpuOps()
    assert ops._records(segs[0]) is None
    outs = kcp.kcp_prefill_local(segs, ops)
    q, k, v = qkv_to_dev(d, cuda_dev)
    o1, S1, _ = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev))
    torch.cuda.synchronize()
    o = torch.cat([x[0] for x in outs])
    assert rel(host(o), host(o1)) < TOL_O and rel(host(outs[-1][1]), host(S1[0])) < TOL_S
    ro, rS, _ = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"])
    assert rel(host(o), ro) < TOL_O and rel(host(outs[-1][1]), rS[0]) < TOL_S
