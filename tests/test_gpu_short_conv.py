"""ShortConv + Swish prologue on the GPU (kda_short_conv, kda_short_conv_step)
against the CPU oracle ("Kimi K3: KDA, attention residuals and Stable
LatentMoE", Sec. 2.1; Swish of Sec. 5)."""
import numpy as np
import pytest
import torch

import oracle
from oracle import prologue
from serving_kda_chunked_gated_gb300 import inputs as I
from kda_testutil import TOL_O, TOL_S, f64, host, rel, to_dev

pytestmark = pytest.mark.gpu

TOL = {torch.bfloat16: TOL_O, torch.float32: 1e-5}


def _inputs(T, C, W, dt, seed, n_seqs):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn((T, C), generator=g).to(dt)
    w = (torch.randn((C, W), generator=g) / W).float()
    b = (0.1 * torch.randn((C,), generator=g)).float()
    s0 = torch.randn((n_seqs, max(W - 1, 0), C), generator=g).float()
    return x, w, b, s0


# packed lengths 0, 1, 2, 147, 250: empty, shorter than the window, crossing the
# 128-token segments of the kernel
CU = [0, 0, 1, 3, 150, 400]


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 4, 8])
def test_short_conv_matches_oracle(kda_lib, cuda_dev, dt, W):
    import serving_kda_chunked_gated_gb300.kda as kda
    C = 256
    x, w, b, s0 = _inputs(CU[-1], C, W, dt, seed=W, n_seqs=len(CU) - 1)
    cu = torch.tensor(CU, dtype=torch.int32)
    for bias, state, act in ((b, s0, True), (None, None, True), (b, s0, False)):
        y, st = kda.short_conv(x.to(cuda_dev), w.to(cuda_dev), None if bias is None else bias.to(cuda_dev),
                               cu_seqlens=cu.to(cuda_dev), state_in=None if state is None else state.to(cuda_dev),
                               activation=act)
        torch.cuda.synchronize()
        ry, rst = prologue.short_conv(x.double().numpy(), w.double().numpy(),
                                      None if bias is None else bias.double().numpy(), cu_seqlens=CU,
                                      state=None if state is None else state.double().numpy(), activation=act)
        assert rel(host(y), ry) < TOL[dt], (bias is None, state is None, act)
        if W > 1:
            assert np.array_equal(st.cpu().numpy(), rst.astype(np.float32))   # the state is copied inputs


def test_decode_steps_continue_the_prefill(kda_lib, cuda_dev):
    import serving_kda_chunked_gated_gb300.kda as kda
    T, C, W = 40, 512, 4
    x, w, b, s0 = _inputs(3 * T, C, W, torch.bfloat16, seed=9, n_seqs=3)
    xs = x.view(3, T, C)                                    # three sequences of T tokens
    cu = torch.tensor([0, T - 5, 2 * (T - 5), 3 * (T - 5)], dtype=torch.int32)
    pre = torch.cat([xs[n, :T - 5] for n in range(3)]).contiguous()
    _, state = kda.short_conv(pre.to(cuda_dev), w.to(cuda_dev), b.to(cuda_dev), cu_seqlens=cu.to(cuda_dev),
                              state_in=s0.to(cuda_dev))
    # states in permuted slots: sequence n lives in row perm[n]
    perm = torch.tensor([2, 0, 1])
    slots_state = torch.empty_like(state)
    slots_state[perm.to(cuda_dev)] = state
    outs = []
    for t in range(T - 5, T):
        xt = xs[:, t].contiguous().to(cuda_dev)
        outs.append(kda.short_conv_step(xt, w.to(cuda_dev), slots_state, bias=b.to(cuda_dev),
                                        slots=perm.to(torch.int32).to(cuda_dev)))
    torch.cuda.synchronize()
    for n in range(3):
        ry, rst = prologue.short_conv(xs[n].double().numpy(), w.double().numpy(), b.double().numpy(),
                                      state=s0[n:n + 1].double().numpy())
        got = torch.stack([o[n] for o in outs]).float().cpu().numpy()
        assert rel(got, ry[T - 5:]) < TOL_O
        assert np.array_equal(slots_state[perm[n]].cpu().numpy(), rst[0].astype(np.float32))


def test_prologue_then_prefill_matches_oracle(kda_lib, cuda_dev):
    """q, k, v pre-activations -> ShortConv + Swish -> KDA prefill (L2Norm on q, k)
    against the oracle's composition of the same steps."""
    import serving_kda_chunked_gated_gb300.kda as kda
    H, d, W = 2, 128, 4
    cu = [0, 70, 300]
    T = cu[-1]
    dd = I.make_prefill(I.workload("prefill_128k", T=T, H=H))
    g = torch.Generator().manual_seed(21)
    pre = [torch.randn((T, H * d), generator=g).to(torch.bfloat16) for _ in range(3)]
    ws = [(torch.randn((H * d, W), generator=g) / W).float() for _ in range(3)]
    cud = torch.tensor(cu, dtype=torch.int32, device=cuda_dev)
    act = [kda.short_conv(p.to(cuda_dev), w.to(cuda_dev), cu_seqlens=cud)[0] for p, w in zip(pre, ws)]
    q, k, v = (a.view(T, H, d) for a in act)
    o, S_T, _ = kda.prefill(q, k, v, to_dev(dd["z"], cuda_dev), to_dev(dd["beta"], cuda_dev),
                            to_dev(dd["A"], cuda_dev), cu_seqlens=cud)
    torch.cuda.synchronize()
    ract = [prologue.short_conv(p.double().numpy(), w.double().numpy(), cu_seqlens=cu)[0] for p, w in zip(pre, ws)]
    # the GPU prefill reads the bf16-rounded prologue outputs; the oracle takes the same rounding
    rq, rk, rv = (torch.from_numpy(a).to(torch.bfloat16).double().numpy().reshape(T, H, d) for a in ract)
    assert rel(host(q.reshape(T, H * d)), ract[0]) < TOL_O
    ro, rS, _ = oracle.prefill(rq, rk, rv, dd["z"], dd["beta"], dd["A"], cu_seqlens=np.array(cu, dtype=np.int32))
    assert rel(host(o), ro) < TOL_O and rel(host(S_T), rS) < TOL_S


def test_full_size_sampled(kda_lib, cuda_dev):
    """131072 tokens x 4096 channels (32 heads x 128), width 4, in 16 packed
    sequences; 64 channels at each end checked against the oracle."""
    import serving_kda_chunked_gated_gb300.kda as kda
    T, C, W = 131072, 4096, 4
    g = torch.Generator(device=cuda_dev).manual_seed(33)
    x = torch.randn((T, C), generator=g, device=cuda_dev).to(torch.bfloat16)
    w = (torch.randn((C, W), generator=g, device=cuda_dev) / W).float()
    b = (0.1 * torch.randn((C,), generator=g, device=cuda_dev)).float()
    cuts = np.sort(np.random.default_rng(34).choice(np.arange(1, T), 15, replace=False))
    cu = np.concatenate([[0], cuts, [T]]).astype(np.int32)
    s0 = torch.randn((16, W - 1, C), generator=g, device=cuda_dev).float()
    y, st = kda.short_conv(x, w, b, cu_seqlens=torch.from_numpy(cu).to(cuda_dev), state_in=s0)
    torch.cuda.synchronize()
    cols = np.r_[0:64, C - 64:C]
    ry, rst = prologue.short_conv(x[:, cols].double().cpu().numpy(), w[cols].double().cpu().numpy(),
                                  b[cols].double().cpu().numpy(), cu_seqlens=cu,
                                  state=s0[:, :, cols].double().cpu().numpy())
    assert rel(y[:, cols].float().cpu().numpy(), ry) < TOL_O
    assert np.array_equal(st[:, :, cols].cpu().numpy(), rst.astype(np.float32))
