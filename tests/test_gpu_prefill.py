"""Prefill on the GPU (kda_prefill through the C ABI) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, parity, qkv_to_dev, rel, to_dev

pytestmark = pytest.mark.gpu


def run_gpu(kda, d, dev, recurrent=False, gate=None, s0=True, alias_state=False):
    q, k, v = qkv_to_dev(d, dev)
    S0 = to_dev(d["S0"], dev) if (s0 and d["S0"] is not None) else None
    g_in = to_dev(d["g_in"], dev, True) if (d["g_in"] is not None and gate is not False) else None
    out = None
    if alias_state and S0 is not None:
        out = {"o": torch.empty_like(v), "S_T": S0,
               "y": torch.empty_like(v) if g_in is not None else None}
    o, S_T, y = kda.prefill(q, k, v, to_dev(d["z"], dev), to_dev(d["beta"], dev), to_dev(d["A"], dev),
                            cu_seqlens=to_dev(d["cu_seqlens"], dev), S0=S0, g_in=g_in,
                            recurrent=recurrent, out=out)
    torch.cuda.synchronize()
    return o, S_T, y


def run_oracle(d, gate=None, s0=True):
    g = f64(d, "g_in") if gate is not False else None
    return oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                          cu_seqlens=d["cu_seqlens"], S0=d["S0"] if s0 else None, g_in=g)


def check(res, ref, tol_o=TOL_O, tol_s=TOL_S, bf16=True, seq_bounds=None):
    o, S_T, y = res
    ro, rS, ry = ref
    parity("o", host(o), ro, tol_o, bf16_out=bf16 and o.dtype == torch.bfloat16, seq_bounds=seq_bounds)
    parity("S_T", host(S_T), rS, tol_s)
    if ry is not None:
        parity("y", host(y), ry, tol_o, bf16_out=True, seq_bounds=seq_bounds, floor_ref=ro)


def test_tiny_fp32(kda_lib, cuda_dev):
    """The tiny workload (T = 64, H = 1, d = 32, fp32, chunk 64 / sub-chunk 16)
    through the chunked form: with its workspace kda_prefill runs the
    chunk-parallel schedule (plan, prep, scan: three launches); the per-token
    kernel (kda_prefill_recurrent) checks the same inputs."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("tiny"))
    ref = run_oracle(d)
    n0 = kda.launch_count()
    res = run_gpu(kda, d, cuda_dev)
    assert kda.launch_count() - n0 == 3            # plan + prep + scan: the chunked form ran
    check(res, ref)
    check(run_gpu(kda, d, cuda_dev, recurrent=True), ref)


@pytest.mark.parametrize("dk", [32, 64])
def test_fp32_small_d_chunked_ragged(kda_lib, cuda_dev, dk):
    """float32 q, k, v with d = 32 and 64 on the chunk-parallel schedule: packed
    ragged sequences (1, 63, 64, 65 and 200 tokens and an empty one), a prefix
    state, snapshots every 64 tokens; against the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    cu = np.array([0, 1, 64, 64, 128, 193, 393], dtype=np.int32)
    H = 2
    d = I.make_prefill(I.workload("tiny", T=int(cu[-1]), H=H, dk=dk, dv=dk, S0_std=0.02, z_std=2.0, A_std=0.5))
    d["cu_seqlens"] = cu
    d["S0"] = (0.02 * np.random.default_rng(11).standard_normal((len(cu) - 1, H, dk, dk))).astype(np.float32)
    q, k, v = qkv_to_dev(d, cuda_dev)
    n0 = kda.launch_count()
    o, S_T, y, snap = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev),
                                  to_dev(d["A"], cuda_dev), cu_seqlens=to_dev(cu, cuda_dev),
                                  S0=to_dev(d["S0"], cuda_dev), snap_interval=64)
    torch.cuda.synchronize()
    assert kda.launch_count() - n0 == 3
    ro, rS, _, rsnap = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                      cu_seqlens=cu, S0=d["S0"], snap_interval=64)
    parity("o", host(o), ro, TOL_O, seq_bounds=cu)
    parity("S_T", host(S_T), rS, TOL_S, seq_bounds=range(len(cu)))
    parity("snapshots", host(snap), rsnap, TOL_S)


@pytest.mark.parametrize("T", [1, 15, 16, 64, 65, 300])
def test_bf16_lengths(kda_lib, cuda_dev, T):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=T, H=2))
    check(run_gpu(kda, d, cuda_dev), run_oracle(d))


def test_bf16_varlen_with_empty_and_single(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("prefill_128k", T=0, H=3, S0_std=0.02)
    d = I.make_prefill(I.workload("prefill_128k", T=400, H=3))
    cu = np.array([0, 0, 1, 130, 130, 400], dtype=np.int32)
    d["cu_seqlens"] = cu
    d["S0"] = (0.02 * np.random.default_rng(1).standard_normal((5, 3, 128, 128))).astype(np.float32)
    check(run_gpu(kda, d, cuda_dev), run_oracle(d))


def test_in_place_state(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=200, H=2))
    check(run_gpu(kda, d, cuda_dev, alias_state=True), run_oracle(d))


@pytest.mark.parametrize("cu", [[0, 700], [0, 0, 1, 64, 130, 130, 400, 1000], [0, 63, 128, 193]])
def test_schedules_agree(kda_lib, cuda_dev, cu):
    """Chunk-parallel (full workspace) and single-pass (minimal workspace)
    schedules: both match the oracle, the error word stays 0, and the two agree
    to rounding."""
    import serving_kda_chunked_gated_gb300.kda as kda
    H = 3
    d = I.make_prefill(I.workload("prefill_128k", T=cu[-1], H=H))
    d["cu_seqlens"] = np.array(cu, dtype=np.int32)
    d["S0"] = (0.02 * np.random.default_rng(7).standard_normal((len(cu) - 1, H, 128, 128))).astype(np.float32)
    q, k, v = qkv_to_dev(d, cuda_dev)
    args = dict(cu_seqlens=to_dev(d["cu_seqlens"], cuda_dev), S0=to_dev(d["S0"], cuda_dev),
                g_in=to_dev(d["g_in"], cuda_dev, True))
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    cu_host = args["cu_seqlens"].cpu()          # kept alive: the args hold its address
    probe = kda.make_prefill_args(q, k, v, z, beta, A, args["cu_seqlens"], cu_host, torch.empty_like(v))
    need = kda.prefill_workspace_size(probe)
    assert need > 4096
    ws_full = torch.zeros(need, dtype=torch.uint8, device=cuda_dev)
    ws_min = torch.zeros(kda.PREFILL_MIN_WORKSPACE, dtype=torch.uint8, device=cuda_dev)
    res = {}
    for name, ws in (("split", ws_full), ("single", ws_min)):
        res[name] = kda.prefill(q, k, v, z, beta, A, workspace=ws, **args)
        torch.cuda.synchronize()
        assert kda.device_error(ws) == kda.KDA_OK, name
    ref = run_oracle(d)
    for name in res:
        check(res[name], ref)
    a, b = res["split"], res["single"]
    assert rel(host(a[0]), host(b[0])) < TOL_O and rel(host(a[1]), host(b[1])) < TOL_S
    assert rel(host(a[2]), host(b[2])) < TOL_O


def test_chunked_matches_recurrent_gpu(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=700, H=4))
    a = run_gpu(kda, d, cuda_dev)
    b = run_gpu(kda, d, cuda_dev, recurrent=True)
    assert rel(host(a[0]), host(b[0])) < TOL_O
    assert rel(host(a[1]), host(b[1])) < TOL_S


def test_adversarial_gates(kda_lib, cuda_dev):
    """Gates at both ends: z = +1e4 (g = g_min every step) and z = -1e4 (no decay)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=260, H=2))
    z = d["z"]
    z[:, 0, :64] = 1e4
    z[:, 0, 64:] = -1e4
    z[::3, 1, :] = 1e4
    check(run_gpu(kda, d, cuda_dev), run_oracle(d))


def test_full_prefill_8k_sampled(kda_lib, cuda_dev):
    """Full 8192-token, 32-head prefill (the prefill_8k workload, chunk-parallel
    schedule); the oracle recomputes three heads."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("prefill_8k")
    d = I.make_prefill(w)
    o, S_T, _ = run_gpu(kda, d, cuda_dev)
    heads = [0, 13, 31]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, _ = run_oracle(ds)
    parity("o", host(o)[:, heads], ro, TOL_O, bf16_out=True)
    parity("S_T", host(S_T)[:, heads], rS, TOL_S)


def test_prefill_128k_bench_config(kda_lib, cuda_dev):
    """The benchmark's headline workload exactly as it is timed: prefill_128k
    (131072 tokens, 32 heads, prefix state S0 ~ N(0, 0.02), fused output gate),
    a full workspace, so the chunk-parallel schedule runs.  o, y and S_T of four
    heads (first and last among them) against the oracle, row by row; two runs
    bit-identical; no bounded wait gave up.  The same inputs through the
    single-pass schedule (minimal workspace) agree with it and with the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("prefill_128k")
    d = I.make_prefill(w)
    q, k, v = qkv_to_dev(d, cuda_dev)
    args = dict(cu_seqlens=to_dev(d["cu_seqlens"], cuda_dev), S0=to_dev(d["S0"], cuda_dev),
                g_in=to_dev(d["g_in"], cuda_dev, True))
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    del d
    o, S_T, y = kda.prefill(q, k, v, z, beta, A, workspace="cache", **args)
    o2, S_T2, y2 = kda.prefill(q, k, v, z, beta, A, workspace="cache", **args)
    torch.cuda.synchronize()
    assert kda.device_error(kda.cached_workspace(cuda_dev)) == 0
    assert torch.equal(o, o2) and torch.equal(S_T, S_T2) and torch.equal(y, y2)
    del o2, S_T2, y2
    kda.release_workspace_cache()
    ws = torch.zeros(4096, dtype=torch.uint8, device=cuda_dev)
    o_sp, S_sp, y_sp = kda.prefill(q, k, v, z, beta, A, workspace=ws, **args)
    torch.cuda.synchronize()
    assert kda.device_error(ws) == 0
    del q, k, v, z, beta, args
    heads = [0, 5, 17, 31]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, ry = run_oracle(ds)
    parity("o", host(o[:, heads]), ro, TOL_O, bf16_out=True)
    parity("y", host(y[:, heads]), ry, TOL_O, bf16_out=True, floor_ref=ro)
    parity("S_T", host(S_T[:, heads]), rS, TOL_S)
    parity("o single-pass", host(o_sp[:, heads[:2]]), ro[:, :2], TOL_O, bf16_out=True)
    parity("S_T single-pass", host(S_sp[:, heads[:2]]), rS[:, :2], TOL_S)
    assert rel(host(o_sp), host(o)) < TOL_O and rel(host(y_sp), host(y)) < TOL_O
    assert rel(host(S_sp), host(S_T)) < TOL_S


def test_full_varlen_16_sampled(kda_lib, cuda_dev):
    """Packed 16-sequence prefill (lengths 512..16384); three heads checked,
    every sequence on its own; the packed result equals per-sequence calls bit
    for bit."""
    import serving_kda_chunked_gated_gb300.kda as kda
    w = I.workload("varlen_16")
    d = I.make_prefill(w)
    o, S_T, _ = run_gpu(kda, d, cuda_dev)
    heads = [0, 16, 31]
    ds = I.make_prefill(w, heads=heads)
    ro, rS, _ = run_oracle(ds)
    cu = d["cu_seqlens"]
    parity("o", host(o)[:, heads], ro, TOL_O, bf16_out=True, seq_bounds=cu)
    parity("S_T", host(S_T)[:, heads], rS, TOL_S, seq_bounds=range(len(cu)))
    for n in (0, 7, 15):
        s, e = int(cu[n]), int(cu[n + 1])
        sub = dict(d)
        for key in ("q", "k", "v", "z", "beta"):
            sub[key] = np.ascontiguousarray(d[key][s:e])
        sub["cu_seqlens"] = np.array([0, e - s], dtype=np.int32)
        o1, S1, _ = run_gpu(kda, sub, cuda_dev)
        assert torch.equal(o1, o[s:e]) and torch.equal(S1[0], S_T[n])


def test_prefill_then_decode_continues_the_sequence(kda_lib, cuda_dev):
    """Prefill 150 tokens on the tensor-core path, then decode 3 more with
    kda_decode_step from its final state: every output matches the oracle's
    single 153-token recurrence (the prefix cache resumes exactly)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=153, H=2))
    T0 = 150
    q, k, v = qkv_to_dev(d, cuda_dev)
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    g_in = to_dev(d["g_in"], cuda_dev, True)
    S0 = to_dev(d["S0"], cuda_dev)
    o, S, y = kda.prefill(q[:T0].contiguous(), k[:T0].contiguous(), v[:T0].contiguous(), z[:T0].contiguous(),
                          beta[:T0].contiguous(), A, S0=S0, g_in=g_in[:T0].contiguous())
    outs, ys = [o], [y]
    for t in range(T0, 153):
        sl = slice(t, t + 1)
        # fresh copies: a one-token slice of a packed tensor is not 16-byte aligned
        od, yd = kda.decode_step(q[sl].clone(), k[sl].clone(), v[sl].clone(), z[sl].clone(),
                                 beta[sl].clone(), A, S, g_in=g_in[sl].clone())
        outs.append(od)
        ys.append(yd)
    torch.cuda.synchronize()
    ro, rS, ry = run_oracle(d)
    assert rel(host(torch.cat(outs)), ro) < TOL_O
    assert rel(host(torch.cat(ys)), ry) < TOL_O
    assert rel(host(S), rS) < TOL_S


def test_split_prefill_resumes_from_state(kda_lib, cuda_dev):
    """prefill(T1) then prefill(T2 | S_T1) equals the oracle on T1 + T2 tokens."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=333, H=2))
    q, k, v = qkv_to_dev(d, cuda_dev)
    z, beta, A = to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev), to_dev(d["A"], cuda_dev)
    S0 = to_dev(d["S0"], cuda_dev)
    c = lambda x, s: x[s].clone()
    a, b = slice(0, 100), slice(100, 333)
    o1, S1, _ = kda.prefill(c(q, a), c(k, a), c(v, a), c(z, a), c(beta, a), A, S0=S0)
    o2, S2, _ = kda.prefill(c(q, b), c(k, b), c(v, b), c(z, b), c(beta, b), A, S0=S1)
    torch.cuda.synchronize()
    ro, rS, _ = run_oracle(d, gate=False)
    assert rel(host(torch.cat([o1, o2])), ro) < TOL_O
    assert rel(host(S2), rS) < TOL_S


def test_options_scale_norm_weight_no_l2norm(kda_lib, cuda_dev):
    """scale != 1, an RMSNorm weight, and qk_l2norm off (inputs pre-normalised)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=130, H=2))
    w = (np.random.default_rng(5).random(128) + 0.5).astype(np.float32)
    q, k, v = qkv_to_dev(d, cuda_dev)
    o, S_T, y = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev),
                            to_dev(d["A"], cuda_dev), S0=to_dev(d["S0"], cuda_dev),
                            g_in=to_dev(d["g_in"], cuda_dev, True), norm_w=to_dev(w, cuda_dev),
                            scale=0.5, qk_l2norm=False)
    torch.cuda.synchronize()
    ro, rS, ry = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"],
                                S0=d["S0"], g_in=f64(d, "g_in"), norm_w=w, scale=0.5, qk_l2norm=False)
    assert rel(host(o), ro) < TOL_O
    assert rel(host(y), ry) < TOL_O
    assert rel(host(S_T), rS) < TOL_S


@pytest.mark.parametrize("T,slab", [(1000, 256), (300, 4096), (12345, 2048)])
def test_prefill_from_host_pipelined(kda_lib, cuda_dev, T, slab):
    """The slab-pipelined host-buffer prefill equals the one-shot device call (slabs
    end on chunk boundaries; the state carries in FP32).  Not bit for bit: each slab
    call picks its own power-of-two scales for the scan's fp16 operands (from its v
    and its S0), and relative fp16 rounding is scale-free only above the subnormal
    range, so entries far below their column's largest may round differently."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=T, H=2))
    pin = lambda x, bf: (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16) if bf
                         else torch.from_numpy(np.ascontiguousarray(x))).pin_memory()
    hq, hk, hv, hg = (pin(d[n], True) for n in ("q", "k", "v", "g_in"))
    hz, hb, hA, hS0 = (pin(d[n], False) for n in ("z", "beta", "A", "S0"))
    o_h, S_h, y_h = kda.prefill_from_host(hq, hk, hv, hz, hb, hA, S0=hS0, g_in=hg, slab=slab)
    torch.cuda.synchronize()
    o, S_T, y = kda.prefill(hq.to(cuda_dev), hk.to(cuda_dev), hv.to(cuda_dev), hz.to(cuda_dev), hb.to(cuda_dev),
                            hA.to(cuda_dev), S0=hS0.to(cuda_dev), g_in=hg.to(cuda_dev))
    torch.cuda.synchronize()
    for name, a_, b_ in (("o", o_h, o), ("y", y_h, y), ("S_T", S_h, S_T)):
        parity(name, host(a_), host(b_.cpu()), 1e-4, row_tol=1e-2)   # a bf16 output may flip one ulp


@pytest.mark.parametrize("case", ["column_spread", "state_dominates_1e3", "state_dominates_1e6", "large_v", "zero_v"])
def test_fp16_operand_range(kda_lib, cuda_dev, case):
    """The chunk-parallel scan multiplies fp16 operands (the tf32 mantissa, a
    narrower range) under power-of-two scaling per value column and per chunk:
    value columns six decades apart (each column checked against its own scale),
    a prefix state a thousand and a million times larger than v that decays
    away, v two thousand times its usual size, and v = 0 (the state only
    decays).  The prefix-state cases check the A tile's per-row power-of-two
    scaling: a row whose decay factors are all small would otherwise sit among
    the fp16 subnormals, and its product with the large state would lose all
    but a few bits (worst y row without the scaling: 1.8e-2 at 1e3, 0.94 at
    1e6)."""
    import serving_kda_chunked_gated_gb300.kda as kda
    d = I.make_prefill(I.workload("prefill_128k", T=300, H=2))
    vf = I.bf16_to_f32(d["v"])
    col = np.ones(128, dtype=np.float64)
    if case == "column_spread":
        col = 10.0 ** np.linspace(-3, 3, 128)
        vf = vf * col.astype(np.float32)
    elif case.startswith("state_dominates"):
        f = 1e6 if case.endswith("1e6") else 1e3
        d["S0"] = (f * np.random.default_rng(5).standard_normal(d["S0"].shape)).astype(np.float32)
    elif case == "large_v":
        vf = vf * 2e3
    else:
        vf = vf * 0.0
        d["S0"] = np.broadcast_to(np.eye(128, dtype=np.float32), d["S0"].shape).copy()
    d["v"] = I.bf16_bits(vf)
    o, S_T, y = run_gpu(kda, d, cuda_dev)
    ro, rS, ry = run_oracle(d)
    parity("o / column scale", host(o) / col, ro / col, TOL_O, bf16_out=True)
    if case.startswith("state_dominates"):
        # once S0 has decayed the outputs are at the scale of v, far below the scale
        # the operands were set for: they keep the same accuracy
        parity("o after the prefix state decayed", host(o)[128:], ro[128:], TOL_O, bf16_out=True)
        # y rows of the first two chunks, each against its own norm (no floor)
        ye = np.linalg.norm(host(y)[:128] - ry[:128], axis=-1) / np.linalg.norm(ry[:128], axis=-1)
        assert ye.max() <= 1e-2, (case, float(ye.max()))
    if case == "zero_v":
        # S_T = the transition applied to S0 = I: one head decays below fp32 over 300
        # tokens; the fp16 record operands carry terms down to 2^-24 of their scale,
        # so the state is exact relative to |S0| once it decays below 2^-14 of it
        for hh in range(2):
            err = np.linalg.norm(host(S_T)[0, hh] - rS[0, hh])
            assert err <= TOL_S * max(np.linalg.norm(rS[0, hh]), 2.0 ** -14 * np.sqrt(128)), (hh, err)
    else:
        parity("S_T / column scale", host(S_T) / col, rS / col, TOL_S)
    if ry is not None:
        parity("y", host(y), ry, TOL_O, bf16_out=True, floor_ref=ro)


def test_prefill_from_host_edge_cases(kda_lib, cuda_dev):
    """kda_prefill_from_host on an empty sequence (S_T = S0, nothing else
    written), on float32 q/k/v with d = 64 in slabs of 64 tokens (a ragged last
    slab), and with a slab longer than the sequence; against kda_prefill on the
    device and the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    pin = lambda x: torch.from_numpy(np.ascontiguousarray(x)).pin_memory()
    # empty sequence: the state passes through
    d = I.make_prefill(I.workload("tiny", T=0, H=2, dk=64, dv=64, S0_std=0.02))
    S0 = (0.02 * np.random.default_rng(3).standard_normal((1, 2, 64, 64))).astype(np.float32)
    empty = lambda shape: torch.empty(shape, dtype=torch.float32).pin_memory()
    o_h, S_h, _ = kda.prefill_from_host(empty((0, 2, 64)), empty((0, 2, 64)), empty((0, 2, 64)), empty((0, 2, 64)),
                                        empty((0, 2)), pin(d["A"]), S0=pin(S0), slab=64)
    torch.cuda.synchronize()
    assert np.array_equal(S_h.numpy(), S0)
    # float32, d = 64, 130 tokens in slabs of 64 and in one slab of 4096
    d = I.make_prefill(I.workload("tiny", T=130, H=2, dk=64, dv=64, S0_std=0.02, z_std=2.0, A_std=0.5))
    S0 = (0.02 * np.random.default_rng(4).standard_normal((1, 2, 64, 64))).astype(np.float32)
    ro, rS, _ = oracle.prefill(f64(d, "q"), f64(d, "k"), f64(d, "v"), d["z"], d["beta"], d["A"], S0=S0)
    q, k, v = qkv_to_dev(d, cuda_dev)
    o_d, S_d, _ = kda.prefill(q, k, v, to_dev(d["z"], cuda_dev), to_dev(d["beta"], cuda_dev),
                              to_dev(d["A"], cuda_dev), S0=to_dev(S0, cuda_dev))
    for slab in (64, 4096):
        o_h, S_h, _ = kda.prefill_from_host(pin(d["q"]), pin(d["k"]), pin(d["v"]), pin(d["z"]), pin(d["beta"]),
                                            pin(d["A"]), S0=pin(S0), slab=slab)
        torch.cuda.synchronize()
        parity(f"o slab {slab}", o_h.numpy(), ro, TOL_O)
        parity(f"S_T slab {slab}", S_h.numpy(), rS, TOL_S)
        parity(f"o slab {slab} vs device call", o_h.numpy(), host(o_d), 1e-4, row_tol=1e-2)
    # bf16 with the fused gate, one slab longer than the sequence
    d = I.make_prefill(I.workload("prefill_128k", T=100, H=2))
    hp = lambda x, bf: (torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16) if bf
                        else torch.from_numpy(np.ascontiguousarray(x))).pin_memory()
    o_h, S_h, y_h = kda.prefill_from_host(hp(d["q"], True), hp(d["k"], True), hp(d["v"], True), hp(d["z"], False),
                                          hp(d["beta"], False), hp(d["A"], False), S0=hp(d["S0"], False),
                                          g_in=hp(d["g_in"], True), slab=16384)
    torch.cuda.synchronize()
    ro, rS, ry = run_oracle(d)
    check((o_h, S_h, y_h), (ro, rS, ry))
