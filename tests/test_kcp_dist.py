"""KDA context parallelism (Sec. 10.2) host logic on CPU ranks (gloo): the
package's KCP driver with oracle-backed per-rank steps reproduces the oracle's
single-pass prefill of the whole sequence on every rank, for uneven segments
and a prefix state."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class OracleOps:
    """KCP steps on the FP64 CPU oracle (per head), torch tensors in and out."""

    def pair(self, seg):
        import oracle
        from oracle import chunked
        H = seg["k"].shape[1]
        Ms, Sts = [], []
        for h in range(H):
            g = oracle.log_decay(seg["z"][:, h].numpy(), float(seg["A"][h]))
            M, St = chunked.kcp_pair(seg["k"][:, h].numpy(), seg["v"][:, h].numpy(), g, seg["beta"][:, h].numpy())
            Ms.append(M)
            Sts.append(St)
        return torch.from_numpy(np.stack(Ms)), torch.from_numpy(np.stack(Sts))

    def apply(self, M, S, St):
        return torch.matmul(M, S) + St

    def prefill(self, seg, S0):
        import oracle
        o, S_T, _ = oracle.prefill(seg["q"].numpy(), seg["k"].numpy(), seg["v"].numpy(), seg["z"].numpy(),
                                   seg["beta"].numpy(), seg["A"].numpy(), S0=S0.numpy()[None], qk_l2norm=False)
        return torch.from_numpy(o), torch.from_numpy(S_T[0]), None


def _sequence(T, H, d, seed):
    rng = np.random.default_rng(seed)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)
    return dict(q=unit(rng.standard_normal((T, H, d))), k=unit(rng.standard_normal((T, H, d))),
                v=rng.standard_normal((T, H, d)), z=2.0 * rng.standard_normal((T, H, d)),
                beta=1 / (1 + np.exp(-rng.standard_normal((T, H)))), A=0.5 * rng.standard_normal(H))


CUTS = {2: [0, 23, 60], 3: [0, 5, 41, 60], 4: [0, 1, 30, 31, 60]}   # uneven, incl. 1-token segments


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import torch.distributed as dist
    from serving_kda_chunked_gated_gb300 import kcp
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        full = _sequence(60, 2, 6, seed=71)
        cuts = CUTS[world]
        seg = {k: torch.from_numpy(np.ascontiguousarray(v[cuts[rank]:cuts[rank + 1]])) if k != "A"
               else torch.from_numpy(v) for k, v in full.items()}
        S_init = torch.from_numpy(0.3 * np.random.default_rng(72).standard_normal((2, 6, 6)))
        from test_kcp_dist import OracleOps
        o, S_T, _ = kcp.kcp_prefill(seg, OracleOps(), S_init=S_init)
        q.put((rank, o.numpy(), S_T.numpy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3, 4])
def test_kcp_ranks_reproduce_the_single_pass(world):
    sys.path.insert(0, ROOT)
    import oracle
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = {r: (o, S) for r, o, S in (q.get(timeout=180) for _ in procs)}
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    full = _sequence(60, 2, 6, seed=71)
    S_init = 0.3 * np.random.default_rng(72).standard_normal((2, 6, 6))
    o_ref, S_ref, _ = oracle.prefill(full["q"], full["k"], full["v"], full["z"], full["beta"], full["A"],
                                     S0=S_init[None], qk_l2norm=False)
    cuts = CUTS[world]
    for r in range(world):
        np.testing.assert_allclose(res[r][0], o_ref[cuts[r]:cuts[r + 1]], rtol=0, atol=1e-11)
    np.testing.assert_allclose(res[world - 1][1], S_ref[0], rtol=0, atol=1e-11)


def test_kcp_local_driver_and_pair_composition():
    """The one-device driver and the pair algebra with the oracle steps."""
    sys.path.insert(0, ROOT)
    import oracle
    from serving_kda_chunked_gated_gb300 import kcp
    full = _sequence(50, 2, 5, seed=73)
    cuts = [0, 12, 13, 50]
    segs = [{k: torch.from_numpy(np.ascontiguousarray(v[cuts[i]:cuts[i + 1]])) if k != "A" else torch.from_numpy(v)
             for k, v in full.items()} for i in range(3)]
    outs = kcp.kcp_prefill_local(segs, OracleOps())
    o_ref, S_ref, _ = oracle.prefill(full["q"], full["k"], full["v"], full["z"], full["beta"], full["A"],
                                     qk_l2norm=False)
    np.testing.assert_allclose(torch.cat([o for o, _, _ in outs]).numpy(), o_ref, rtol=0, atol=1e-11)
    np.testing.assert_allclose(outs[-1][1].numpy(), S_ref[0], rtol=0, atol=1e-11)
    # (M2, S2) o (M1, S1) = (M2 M1, S2 + M2 S1): composing the first two pairs
    ops = OracleOps()
    (M1, S1), (M2, S2) = ops.pair(segs[0]), ops.pair(segs[1])
    seg12 = {k: torch.cat([segs[0][k], segs[1][k]]) if k != "A" else segs[0][k] for k in segs[0]}
    M12, S12 = ops.pair(seg12)
    np.testing.assert_allclose(torch.matmul(M2, M1).numpy(), M12.numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(ops.apply(M2, S1, S2).numpy(), S12.numpy(), rtol=0, atol=1e-12)


def _fake_seg(dtype, T=3, H=2, d=128):
    seg = {key: torch.zeros((T, H, d), dtype=dtype) for key in ("q", "k")}
    seg["v"] = torch.ones((T, H, d), dtype=dtype)
    seg.update(z=torch.zeros((T, H, d)), beta=torch.zeros((T, H)), A=torch.zeros(H))
    return seg


def test_gpu_ops_share_one_set_of_records_per_segment(monkeypatch):
    """GpuOps builds a segment's chunk records once: the pair is two scans over
    them (M with the zero-v flag from S0 = I, S~ from zero), the segment's
    outputs a third; the records are released after it.  Inputs without a
    chunk-parallel schedule (fp32) take three kda_prefill calls instead."""
    sys.path.insert(0, ROOT)
    from serving_kda_chunked_gated_gb300 import kcp, kda
    calls = []

    def fake_records(q, k, v, z, beta, A, **kw):
        calls.append(("records",))
        return object()

    def fake_scan(rec, S0=None, g_in=None, norm_w=None, want_o=True, want_state=True, zero_v=False, **kw):
        H, d = 2, 128
        eye = S0 is not None and torch.equal(S0[0, 0], torch.eye(d))
        calls.append(("scan", zero_v, eye, S0 is None, want_o))
        return (torch.zeros((3, H, d)) if want_o else None), torch.zeros((1, H, d, d)), None

    def fake_prefill(q, k, v, z, beta, A, S0=None, want_o=True, **kw):
        calls.append(("prefill", bool((v == 0).all()), S0 is not None, want_o))
        H, d = q.shape[1], q.shape[2]
        return (torch.zeros((3, H, d)) if want_o else None), torch.zeros((1, H, d, d)), None

    monkeypatch.setattr(kda, "prefill_records", fake_records)
    monkeypatch.setattr(kda, "prefill_scan", fake_scan)
    monkeypatch.setattr(kda, "prefill", fake_prefill)
    ops = kcp.GpuOps()
    seg = _fake_seg(torch.bfloat16)
    M, St = ops.pair(seg)
    assert M.shape == (2, 128, 128) and St.shape == (2, 128, 128)
    ops.prefill(seg, torch.zeros((2, 128, 128)))
    assert calls == [("records",), ("scan", True, True, False, False), ("scan", False, False, True, False),
                     ("scan", False, False, False, True)]
    assert ops._rec == {}
    calls.clear()
    seg32 = _fake_seg(torch.float32, d=64)
    ops.pair(seg32)
    ops.prefill(seg32, torch.zeros((2, 64, 64)))
    assert calls == [("prefill", True, True, False), ("prefill", False, False, False), ("prefill", False, True, True)]
